// gemm.cu -- block-scaled FP8 GEMM (dense and grouped) for sm_103a.
//
//   y[m,n] = bf16( sum_kb fp32(sx[m,kb] * sw[n/128,kb]) * P_kb[m,n] )
//
// ("DeepSeek-V3" repository overview, section "FP8 混合精度训练": fp8_gemm of
// the per-token/128-channel quantised activations with the 128x128
// block-quantised weights; fp32 promotion once per 128-wide K chunk after
// four K=32 MMAs, after the Float8 paragraph of the 88811315.cn post and the
// "FP8 量化" section of the qdgithub overview.)
//
// Design (one persistent CTA per SM, warp-specialised; 384 threads for 160-
// and 256-column tiles, 512 for 192-column tiles):
//   warp 0      TMA producer: A (128 x 128 B) and B (BN x 128 B) tiles of one
//               K chunk per pipeline stage, 128-byte swizzled, mbarrier
//               completion by byte count.
//   warps 1-2   MMA issuers taking alternate chunks (warp 1 also owns the
//               TMEM allocation): per chunk, four tcgen05.mma.kind::f8f6f4
//               (M=128, N=BN, K=32) into one of 512/BN TMEM buffers of BN
//               fp32 columns, then tcgen05.commit to free the smem stage and
//               to publish the chunk.  A thread issuing MMAs is held back
//               until the tensor core takes them, so with one issuer the
//               tensor core idled through that thread's two barrier waits
//               every chunk; with two, one warp waits while the other
//               issues.  Chunks use separate buffers and stages, and each
//               commit tracks only its own thread's MMAs, so the two
//               streams need no ordering between them.
//   warp 3      scale loader: per block of four chunks, the tile's sx
//               (128 rows x 4 chunks, one 16-byte TMA box column per row)
//               and the at most three weight-scale rows the tile touches,
//               into a ring of four slots (sfull/sempty mbarriers).  Having
//               every promotion thread fetch its own row's sx from global
//               memory, 4 scattered bytes per chunk, cost up to a third of
//               the large GEMMs' time in load/store traffic.
//   warps 4-    promotion + epilogue: two warpgroups (three for 192-column
//               tiles), each owning BN/NWG columns; thread = one row (TMEM
//               lane).  Per chunk:
//               tcgen05.ld the raw chunk sum P_kb, acc += fp32(sx*sw) * P_kb
//               in registers (packed f32x2 FMAs), release the TMEM buffer.
//               After the last chunk of a tile: round to bf16 and store (or
//               store fp32 partials for split-K).
// Every promotion thread keeps BN/NWG fp32 accumulators (128 at BN = 256),
// so the warpgroups rebalance registers after set-up (setmaxnreg): the
// set-up warpgroup drops to Roles::kRegsSetup, the promotion warpgroups rise
// to Roles::kRegsPromo.  Per SM sub-partition (one set-up warp + NWG
// promotion warps) that stays within the (1 + NWG) * Roles::kRegsLaunch
// registers per lane the launch reserved; the host refuses the kernel unless
// its compiled register count is Roles::kRegsLaunch.
// The TMEM buffers let the tensor core run up to 512/BN - 1 chunks ahead of
// the CUDA cores that promote them.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "codec.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

constexpr int BM = 128;           // tile rows (tokens) = TMEM lanes
constexpr int BK = 128;           // K chunk = one scale block = 4 MMAs of K=32
constexpr int UMMA_K = 32;
constexpr int kMmaWarp0 = 1;      // MMA issuers: warps 1 and 2
constexpr int kMmaWarps = 2;
constexpr int kEpiWarp0 = 4;      // first promotion/epilogue warp
constexpr int kScaleWarp = 3;     // scale loader

// Promotion warpgroups per tile width: two for 160- and 256-column tiles,
// three for 192, whose warpgroups then hold 64 columns each and load a
// chunk's share from TMEM in one go.  The set-up warpgroup (warps 0-3) gives
// registers to the promotion warpgroups with setmaxnreg; per SM
// sub-partition one set-up warp and NWG promotion warps must fit in the
// (1 + NWG) * kRegsLaunch registers per lane the launch reserved.
__host__ __device__ constexpr int nwg_for(int bn) { return bn == 192 ? 3 : 2; }
template <int NWG>
struct Roles {
    static constexpr int kThreads = 128 * (1 + NWG);
    static constexpr int kEpiWarps = 4 * NWG;
    static constexpr int kRegsLaunch = NWG == 2 ? 168 : 128;  // 65536 / threads, a multiple of 8
    static constexpr int kRegsSetup = NWG == 2 ? 56 : 40;
    static constexpr int kRegsPromo = NWG == 2 ? 224 : 152;
    static_assert(kRegsLaunch * kThreads <= 65536, "one CTA per SM");
    static_assert(kRegsSetup + NWG * kRegsPromo <= (1 + NWG) * kRegsLaunch, "register split must fit the launch");
};
constexpr int kScaleChunks = 4;   // K chunks per scale block (one 16-byte TMA column of sx)
constexpr int kScaleSlots = 4;    // scale blocks in flight
constexpr int kSwBlocks = 3;      // weight-scale blocks a tile of <= 256 columns can touch
constexpr int kGroupM = 16;       // dense raster: 16 m-tiles share a sweep over n
constexpr int kMaxGroups = 1024;

template <int BN, int STAGES>
struct Layout {
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = STAGES * A_BYTES;
    // TMEM chunk buffers, each starting on a 32-column boundary
    static constexpr int BUF_COLS = (BN + 31) / 32 * 32;
    static constexpr int NBUF = 512 / BUF_COLS;
    // full[S], empty[S], tfull[NBUF], tempty[NBUF], done[2], sfull[4], sempty[4]
    static constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
    // + one drain barrier per issuer + sfull/sempty per scale slot
    // ... + hbar[2] (SwiGLU FP8 output: the two warpgroups' row amaxes, by tile parity)
    static constexpr int NUM_BARS = 2 * STAGES + 2 * NBUF + kMmaWarps + 2 * kScaleSlots + 2;
    static constexpr int OFF_TMEM = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM + 4;
    static constexpr int OFF_TABLE = (OFF_ABORT + 4 + 15) & ~15;  // grouped: tile prefix [G+1]
    static constexpr int TABLE_BYTES = (kMaxGroups + 1) * 4;
    // scale slots: sx of the tile's 128 rows x kScaleChunks chunks (the TMA
    // box, row-major), then the weight scales of kSwBlocks blocks x chunks
    static constexpr int SX_SLOT = BM * kScaleChunks * 4;
    static constexpr int SW_SLOT = kSwBlocks * kScaleChunks * 4;
    static constexpr int OFF_SX = (OFF_TABLE + TABLE_BYTES + 127) & ~127;
    static constexpr int OFF_SWS = OFF_SX + kScaleSlots * SX_SLOT;
    // fused bias: per scale slot, the bf16 bias of the tile's BN columns
    // (written with the first scale block of each tile)
    static constexpr int OFF_BIAS = (OFF_SWS + kScaleSlots * SW_SLOT + 15) & ~15;
    static constexpr int BIAS_SLOT = BN * 2;
    static constexpr int BIAS_BYTES = kScaleSlots * BIAS_SLOT;
    // SwiGLU FP8 output: per tile parity, per warpgroup, the amax of each row's 64 values
    static constexpr int OFF_HAMAX = OFF_BIAS + BIAS_BYTES;
    static constexpr int HAMAX_BYTES = 2 * 2 * BM * 4;
    // bf16 output staging of 256-column tiles: per promotion warp two 1 KB
    // boxes (32 rows x 16 columns, 32-byte swizzle) that TMA stores drain
    static constexpr int EPI_WARPS = BN == 256 ? 8 : 0;
    static constexpr int OFF_EPI = (OFF_HAMAX + HAMAX_BYTES + 1023) & ~1023;
    static constexpr int EPI_BYTES = EPI_WARPS * 2 * 1024;
    // weight gradient (160-column tiles): per scale slot the column factors
    // of the tile's BN columns for kScaleChunks token chunks ([chunk][column])
    static constexpr int CF_SLOT = BN == 160 ? kScaleChunks * BN * 4 : 0;
    static constexpr int OFF_CF = (OFF_EPI + EPI_BYTES + 127) & ~127;
    static constexpr int BYTES = OFF_CF + kScaleSlots * CF_SLOT;
    static constexpr int ALLOC = BYTES + 1024;                    // slack to align the base to 1024
    static constexpr uint32_t TMEM_COLS = 512;                  // allocation: a power of two
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms need 1024-byte alignment");
    static_assert(NBUF >= 2 && NBUF * BUF_COLS <= 512, "two or more chunk buffers must fit in TMEM");
    static_assert(ALLOC <= 227 * 1024, "shared memory per CTA");
};

struct Params {
    const float* sx;
    int64_t lds;
    const float* sw;
    uint16_t* y;             // bf16 output, or nullptr when only yq is written
    int64_t ldy;
    // fused epilogue (dense, 256-column tiles for yq): y += bias before the
    // bf16 rounding; yq / sy = the bf16 output quantised per row per 128
    // columns, as act_quant would quantise it
    const uint16_t* bias;    // bf16 [N] or nullptr
    const float* sw3;        // SwiGLU grouped: w3's weight scales (p.sw holds w1's)
    uint8_t* yq;             // e4m3 [M, ldyq] or nullptr
    int64_t ldyq;
    float* sy;               // fp32 [M, ldsy]
    int64_t ldsy;
    const int32_t* offsets;  // grouped: device [G+1], else nullptr
    int G;
    int M, N, KB;
    int MT, NT;              // dense: m-tiles, n-tiles
    int num_tiles;           // dense: MT * NT (x splits for split-K)
    // split-K: each tile's K chunks are cut into `splits` ranges of `kps`
    // chunks; split s writes fp32 partial sums to partial[s][M][N]
    int splits, kps;
    float* partial;
    // weight gradient: dW [M, ldyf] fp32 (M = output rows, N = output columns,
    // KB = token chunks)
    float* yf;
    int64_t ldyf;
    unsigned* err;
    uint64_t timeout_ns;
};

struct Tile {
    int tile;    // tile index
    int m0;      // first row of A / y
    int m_end;   // one past the last valid row
    int n0;      // first output column
    int b_row;   // first row of the B operand (g * N + n0 for grouped)
    int sw_base; // first weight-scale row of the operand (g * NB for grouped, else 0)
    int kb0, kb1;  // chunk range of this piece of the tile
};

template <int BN>
__device__ __forceinline__ Tile dense_tile(const Params& p, int t) {
    Tile tl;
    tl.tile = t;
    const int per_group = kGroupM * p.NT;
    const int grp = t / per_group;
    const int first_m = grp * kGroupM;
    const int gm = min(p.MT - first_m, kGroupM);
    const int local = t - grp * per_group;
    const int mt = first_m + local % gm;
    const int nt = local / gm;
    tl.m0 = mt * BM;
    tl.m_end = min(p.M, tl.m0 + BM);
    tl.n0 = nt * BN;
    tl.b_row = tl.n0;
    tl.sw_base = 0;
    tl.kb0 = 0;
    tl.kb1 = p.KB;
    return tl;
}

// prefix[g] = number of tiles of experts < g; tile t belongs to the last
// expert g with prefix[g] <= t (empty experts have prefix[g] == prefix[g+1]).
template <int BN>
__device__ __forceinline__ Tile grouped_tile(const Params& p, const int* prefix, int t) {
    int lo = 0, hi = p.G;  // invariant: prefix[lo] <= t < prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= t) lo = mid; else hi = mid;
    }
    const int g = lo;
    const int r0 = min(max(__ldg(p.offsets + g), 0), p.M);
    const int r1 = min(max(__ldg(p.offsets + g + 1), r0), p.M);
    const int mtiles = max((r1 - r0 + BM - 1) / BM, 1);
    const int local = t - prefix[g];
    const int mt = local % mtiles;
    const int nt = local / mtiles;
    Tile tl;
    tl.tile = t;
    tl.m0 = r0 + mt * BM;
    tl.m_end = r1;
    tl.n0 = nt * BN;
    tl.b_row = g * p.N + tl.n0;
    tl.sw_base = g * ((p.N + 127) / 128);
    tl.kb0 = 0;
    tl.kb1 = p.KB;
    return tl;
}

// Warp-wide exclusive scan of per-expert tile counts into prefix[0..G].
template <int BN>
__device__ void build_tile_table(const Params& p, int* prefix, int lane) {
    const int per = (p.G + 31) / 32;
    const int g0 = lane * per;
    const int nt = (p.N + BN - 1) / BN;
    int local = 0;
    for (int i = 0; i < per; ++i) {
        const int g = g0 + i;
        if (g < p.G) {
            const int r0 = min(max(__ldg(p.offsets + g), 0), p.M);
            const int r1 = min(max(__ldg(p.offsets + g + 1), r0), p.M);
            local += ((r1 - r0 + BM - 1) / BM) * nt;
        }
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
        const int g = g0 + i;
        if (g < p.G) {
            prefix[g] = run;
            const int r0 = min(max(__ldg(p.offsets + g), 0), p.M);
            const int r1 = min(max(__ldg(p.offsets + g + 1), r0), p.M);
            run += ((r1 - r0 + BM - 1) / BM) * nt;
        }
    }
    if (lane == 31) prefix[p.G] = incl;
}

// Wait used while draining in-flight async work before the CTA exits: it
// ignores the abort flag (the work must land before its memory is released)
// but keeps the time limit.
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
    int no_abort = 0;
    WaitCtl c2{&no_abort, ctl.err, ctl.timeout_ns};
    const bool ok = bounded_wait(bar, parity, c2);
    __syncwarp();
    return ok;
}

// MODE: how tiles map to work.
// kGroupedSwiglu: grouped, each tile = 128 columns of w1 (gate) next to the
// same 128 columns of w3 (up), output h = silu(gate) * up.
// kWgrad: the weight gradient dW = dY^T X contracting over tokens; the
// operands are the column-quantised dY^T and X^T (token-contiguous rows), and
// the promotion factor of chunk kb (128 tokens) for output (n, k) is
// RN(sdy[kb][n] * sx[kb][k]), a row factor times a column factor.
enum : int { kDense = 0, kSplitK = 1, kGrouped = 2, kGroupedSwiglu = 3, kWgrad = 4 };
__host__ __device__ constexpr bool is_grouped(int mode) { return mode == kGrouped || mode == kGroupedSwiglu; }
// output columns one tile covers: BN, or 128 h columns for SwiGLU tiles
template <int BN, int MODE>
__host__ __device__ constexpr int tile_cols() { return MODE == kGroupedSwiglu ? 128 : BN; }

// Walks the work of one CTA: tiles strided over the grid; for split-K the
// work unit is (tile, split) and covers the split's range of K chunks.
template <int BN, int MODE>
struct WorkCursor {
    int t;
    __device__ __forceinline__ void begin(const Params&) { t = blockIdx.x; }
    __device__ __forceinline__ bool next(const Params& p, const int* prefix, int num_tiles, Tile& tl) {
        if (t >= num_tiles) return false;
        if (is_grouped(MODE)) {
            tl = grouped_tile<tile_cols<BN, MODE>()>(p, prefix, t);
        } else if (MODE == kSplitK) {
            const int split = t % p.splits;
            tl = dense_tile<BN>(p, t / p.splits);
            tl.tile = split;  // for split-K the piece's index is its split
            tl.kb0 = split * p.kps;
            tl.kb1 = min(p.KB, tl.kb0 + p.kps);
        } else {
            tl = dense_tile<BN>(p, t);
        }
        t += gridDim.x;
        return true;
    }
};

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int BN, int STAGES, int MODE>
__global__ void __launch_bounds__(Roles<nwg_for(BN)>::kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB3, const __grid_constant__ CUtensorMap tmS,
                    const __grid_constant__ CUtensorMap tmY, const __grid_constant__ Params p) {
    using L = Layout<BN, STAGES>;
    using R = Roles<nwg_for(BN)>;
    constexpr int kEpiWarps = R::kEpiWarps;
    static_assert(BN == 160 || BN == 192 || BN == 256, "tile widths the host dispatches");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
    const uint32_t sbase = smem_u32(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const uint32_t bar0 = sbase + L::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    constexpr int NBUF = L::NBUF;
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + NBUF + b); };
    auto done_bar = [&](int w) { return bar0 + 8u * (2 * STAGES + 2 * NBUF + w); };
    auto sfull_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 2 * NBUF + kMmaWarps + s); };
    auto sempty_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 2 * NBUF + kMmaWarps + kScaleSlots + s); };
    auto h_bar = [&](int par) { return bar0 + 8u * (2 * STAGES + 2 * NBUF + kMmaWarps + 2 * kScaleSlots + par); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_ABORT);
    int* prefix = reinterpret_cast<int*>(smem + L::OFF_TABLE);

    if (threadIdx.x == 32) {  // the descriptors are kernel parameters: fetch them while the set-up runs
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (MODE == kGroupedSwiglu || MODE == kWgrad) tma_prefetch_desc(&tmB3);
        tma_prefetch_desc(&tmS);
        if (BN == 256 && (MODE == kDense || MODE == kGrouped) && p.y != nullptr) tma_prefetch_desc(&tmY);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < NBUF; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), kEpiWarps);
        }
        for (int w = 0; w < kMmaWarps; ++w) mbar_init(done_bar(w), 1);
        for (int s = 0; s < kScaleSlots; ++s) {
            mbar_init(sfull_bar(s), 1 + 32);  // the TMA's byte count + one arrival per loader lane
            mbar_init(sempty_bar(s), kEpiWarps);
        }
        for (int par = 0; par < 2; ++par) mbar_init(h_bar(par), kEpiWarps);
        *abort_flag = 0;
        fence_barrier_init();
    }
    // Everything above touches only shared memory; from here on the kernel
    // reads its inputs and claims TMEM, which the previous kernel in the
    // stream may still be using.
    grid_dependency_wait();
    allow_dependents();
    if (warp == 1) tmem_alloc(sbase + L::OFF_TMEM, L::TMEM_COLS);
    constexpr bool GROUPED = is_grouped(MODE);
    constexpr bool SWIGLU = MODE == kGroupedSwiglu;
    // bf16 output of 256-column dense / grouped tiles leaves through shared
    // memory and TMA stores (whole 32-row boxes; rows past M are dropped by
    // the tensor map, rows past a grouped expert's end take the direct path)
    constexpr bool TMA_EPI = BN == 256 && (MODE == kDense || MODE == kGrouped);
    static_assert(!SWIGLU || BN == 256, "SwiGLU tiles are 128 gate + 128 up columns");
    if (GROUPED && warp == kEpiWarp0) build_tile_table<tile_cols<BN, MODE>()>(p, prefix, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::OFF_TMEM);
    const int num_tiles = GROUPED ? prefix[p.G] : p.num_tiles;
    const WaitCtl ctl{abort_flag, p.err, p.timeout_ns};



    if (warp < kEpiWarp0) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R::kRegsSetup));
      if (warp == 0) {
        // ------------------------------------------------------------ producer
        uint32_t it = 0;
        bool ok = true;
        WorkCursor<BN, MODE> wc;
        wc.begin(p);
        Tile tl;
        // One lane runs the loop: its waits and the TMA issues are single-
        // thread operations, and a lone lane polls a barrier with less
        // overhead than a warp-wide vote.
        if (lane == 0) {
            while (ok && wc.next(p, prefix, num_tiles, tl)) {
                for (int kb = tl.kb0; kb < tl.kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!bounded_wait(empty_bar(s), ph ^ 1u, ctl)) { ok = false; break; }
                    mbar_arrive_expect_tx(full_bar(s), L::STAGE_BYTES);
                    tma_load_2d(sbase + L::OFF_A + s * L::A_BYTES, &tmA, full_bar(s), kb * BK, tl.m0);
                    if constexpr (SWIGLU) {  // gate rows, then the same rows of w3
                        tma_load_2d(sbase + L::OFF_B + s * L::B_BYTES, &tmB, full_bar(s), kb * BK, tl.b_row);
                        tma_load_2d(sbase + L::OFF_B + s * L::B_BYTES + 128 * BK, &tmB3, full_bar(s), kb * BK,
                                    tl.b_row);
                    } else {
                        tma_load_2d(sbase + L::OFF_B + s * L::B_BYTES, &tmB, full_bar(s), kb * BK, tl.b_row);
                    }
                }
            }
        }
        __syncwarp();
        it = __shfl_sync(0xffffffffu, it, 0);
        // Every issued load must land before the CTA's shared memory goes away.
        const uint32_t first = it > STAGES ? it - STAGES : 0;
        for (uint32_t j = first; j < it; ++j) drain_wait(full_bar(j % STAGES), (j / STAGES) & 1u, ctl);
    } else if (warp < kMmaWarp0 + kMmaWarps) {
        // ------------------------------------------------------------ MMA issuers
        constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
        const uint32_t mw = static_cast<uint32_t>(warp - kMmaWarp0);  // takes chunks with it % 2 == mw
        uint32_t it = 0;
        bool ok = true, issued = false;
        WorkCursor<BN, MODE> wc;
        wc.begin(p);
        Tile tl;
        if (lane == 0) {  // one lane runs the loop (single-thread waits, MMAs and commits)
            while (ok && wc.next(p, prefix, num_tiles, tl)) {
                for (int kb = tl.kb0; kb < tl.kb1; ++kb, ++it) {
                    if ((it % kMmaWarps) != mw) continue;
                    const int s = it % STAGES;
                    const uint32_t sph = (it / STAGES) & 1u;
                    const int b = it % NBUF;
                    const uint32_t bph = (it / NBUF) & 1u;
                    if (!bounded_wait(tempty_bar(b), bph ^ 1u, ctl)) { ok = false; break; }
                    if (!bounded_wait(full_bar(s), sph, ctl)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t adesc = sdesc_kmajor_sw128(sbase + L::OFF_A + s * L::A_BYTES);
                    const uint64_t bdesc = sdesc_kmajor_sw128(sbase + L::OFF_B + s * L::B_BYTES);
                    const uint32_t d = tmem + static_cast<uint32_t>(b * L::BUF_COLS);
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)  // +32 bytes along K = +2 in the address field
                        umma_e4m3(d, adesc + 2u * k, bdesc + 2u * k, idesc, k > 0 ? 1u : 0u);
                    umma_commit(empty_bar(s));
                    umma_commit(tfull_bar(b));
                    issued = true;
                }
            }
            // All of this warp's MMAs must finish before TMEM is released.
            if (issued) umma_commit(done_bar(mw));
        }
        __syncwarp();
        if (__shfl_sync(0xffffffffu, issued ? 1 : 0, 0)) drain_wait(done_bar(mw), 0, ctl);
      } else if (warp == kScaleWarp) {
        // ------------------------------------------------------------ scale loader
        // Per block of kScaleChunks chunks: sx of the tile's rows by TMA (one
        // 16-byte column per row, so the promotion threads never gather
        // scattered 4-byte values), and the tile's weight scales by plain loads.
        const int nblk = (p.N + 127) / 128;  // weight-scale blocks per operand
        float* sw_slots = reinterpret_cast<float*>(smem + L::OFF_SWS);
        uint32_t sb = 0;
        bool ok = true;
        WorkCursor<BN, MODE> wc;
        wc.begin(p);
        Tile tl;
        while (ok && wc.next(p, prefix, num_tiles, tl)) {
            const int fb = tl.n0 / 128;      // the tile's first weight-scale block
            // lane (bi, c) of the first kSwBlocks * kScaleChunks lanes loads the
            // weight scale of block fb + bi, chunk c of a scale block; blocks
            // past N and chunks past K are never used and read as 0
            const int bi = lane / kScaleChunks;
            bool sw_lane;
            const float* swr;
            if constexpr (MODE == kWgrad) {  // no weight scales: both factors come by TMA
                sw_lane = false;
                swr = nullptr;
            } else if constexpr (SWIGLU) {  // slot rows 0 and 1: the tile's w1 and w3 blocks
                sw_lane = lane < 2 * kScaleChunks && fb < nblk;
                swr = (bi == 0 ? p.sw : p.sw3) + static_cast<int64_t>(tl.sw_base + fb) * p.KB;
            } else {
                sw_lane = lane < kSwBlocks * kScaleChunks && fb + bi < nblk;
                swr = p.sw + static_cast<int64_t>(tl.sw_base + (sw_lane ? fb + bi : 0)) * p.KB;
            }
            auto load_sw = [&](int q) {
                const int kb = q * kScaleChunks + lane % kScaleChunks;
                return sw_lane && kb < p.KB ? __ldg(swr + kb) : 0.0f;
            };
            const int q1 = (tl.kb1 - 1) / kScaleChunks;
            float v = load_sw(tl.kb0 / kScaleChunks);
            // fused bias: lane l takes the tile's columns l, l + 32, ...;
            // loaded now (alongside the first weight scales), stored with the
            // tile's first scale block; columns past N read as 0
            constexpr int kBiasPerLane = BN / 32;
            uint16_t bias_v[kBiasPerLane];
#pragma unroll
            for (int i = 0; i < kBiasPerLane; ++i) {
                const int n = tl.n0 + lane + 32 * i;
                bias_v[i] = (p.bias != nullptr && n < p.N) ? p.bias[n] : uint16_t{0};
            }
            for (int q = tl.kb0 / kScaleChunks; q <= q1; ++q, ++sb) {
                // the next block's weight scales load while this block waits for its slot
                const float v_next = q < q1 ? load_sw(q + 1) : 0.0f;
                const int s = sb % kScaleSlots;
                const uint32_t ph = (sb / kScaleSlots) & 1u;
                if (!warp_wait(sempty_bar(s), ph ^ 1u, ctl)) { ok = false; break; }
                if (lane == 0) {
                    if constexpr (MODE == kWgrad) {
                        // row factors sdy[chunk][n] of the tile's 128 rows and
                        // column factors sx[chunk][k] of its BN columns, for
                        // kScaleChunks token chunks each
                        mbar_arrive_expect_tx(sfull_bar(s), L::SX_SLOT + L::CF_SLOT);
                        tma_load_2d(sbase + L::OFF_SX + s * L::SX_SLOT, &tmS, sfull_bar(s), tl.m0, q * kScaleChunks);
                        tma_load_2d(sbase + L::OFF_CF + s * L::CF_SLOT, &tmB3, sfull_bar(s), tl.n0, q * kScaleChunks);
                    } else {
                        mbar_arrive_expect_tx(sfull_bar(s), L::SX_SLOT);
                        tma_load_2d(sbase + L::OFF_SX + s * L::SX_SLOT, &tmS, sfull_bar(s), q * kScaleChunks, tl.m0);
                    }
                }
                if (lane < kSwBlocks * kScaleChunks) sw_slots[s * (kSwBlocks * kScaleChunks) + lane] = v;
                if (p.bias != nullptr && q == tl.kb0 / kScaleChunks) {
                    uint16_t* bias_slot = reinterpret_cast<uint16_t*>(smem + L::OFF_BIAS + s * L::BIAS_SLOT);
#pragma unroll
                    for (int i = 0; i < kBiasPerLane; ++i) bias_slot[lane + 32 * i] = bias_v[i];
                }
                mbar_arrive(sfull_bar(s));   // releases this lane's stores
                v = v_next;
            }
        }
        // Every issued sx load must land before the CTA's shared memory goes away.
        const uint32_t first = sb > kScaleSlots ? sb - kScaleSlots : 0;
        for (uint32_t j = first; j < sb; ++j)
            drain_wait(sfull_bar(j % kScaleSlots), (j / kScaleSlots) & 1u, ctl);
      }
    } else {
        // ------------------------------------------------------------ promotion + epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R::kRegsPromo));
        constexpr int COLS = BN / nwg_for(BN);  // columns per warpgroup
        // A warpgroup holding 64 or 80 columns loads its share of a chunk at
        // once and releases the TMEM buffer before its FMAs (WHOLE); with 128
        // columns (no room for 128 more registers) it walks 16-column slices,
        // loading slice c+1 during slice c's FMAs, and releases at the end.
        constexpr bool WHOLE = COLS <= 96;
        constexpr int SW = 16;
        static_assert(COLS % 16 == 0, "promotion columns come in 16-column slices");
        constexpr int NCH = COLS / SW;      // 16-column slices (and scale groups) per warpgroup
        constexpr int SP = SW / 2;          // packed pairs per slice
        // A warpgroup's columns (at most 128) touch at most two 128-column
        // weight-scale blocks; each 16-column slice lies inside one of them.
        static_assert(COLS <= 128 && 128 % SW == 0, "slice-to-scale-block mapping");
        // Tiles of 256 columns start on a block boundary, so each warpgroup's
        // 128 columns share one weight scale per chunk.
        constexpr bool ONE_BLOCK = COLS == 128 && BN % 128 == 0 && !SWIGLU;
        // SwiGLU tiles: a warpgroup's 8 slices are 64 gate columns (w1's
        // scale) then the same 64 columns of up (w3's scale), 128 TMEM
        // columns apart.
        constexpr int NF = SWIGLU ? 2 : ONE_BLOCK ? 1 : NCH;  // distinct scale factors per chunk
        auto fsel = [](int c) { return SWIGLU ? (c >= NCH / 2 ? 1 : 0) : ONE_BLOCK ? 0 : c; };
        auto slice_col = [](int c) { return SW * c + (SWIGLU && c >= NCH / 2 ? 64 : 0); };
        const int ew = warp - kEpiWarp0;
        const int wg = ew >> 2;
        const int quarter = warp & 3;       // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const int col0 = SWIGLU ? wg * 64 : wg * COLS;  // first TMEM column of the warpgroup
        const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
        // Scales come from the loader's slots (sfull/sempty per block of
        // kScaleChunks chunks).
        const float* sx_slots = reinterpret_cast<const float*>(smem + L::OFF_SX);
        const float* sw_slots = reinterpret_cast<const float*>(smem + L::OFF_SWS);
        uint32_t ss = 0;                    // scale blocks consumed
        uint32_t h_tiles = 0;               // SwiGLU FP8 output: tiles exchanged (barrier parity, phase)
        uint32_t epi_n = 0;                 // TMA-store epilogue: boxes this warp has stored
        uint32_t it = 0;
        bool ok = true;
        WorkCursor<BN, MODE> wc;
        wc.begin(p);
        Tile tl;
        while (ok && wc.next(p, prefix, num_tiles, tl)) {
            const int m = tl.m0 + row;
            const bool row_ok = m < tl.m_end;
            // The warpgroup's columns [n_first, n_last] lie in weight-scale
            // blocks i0 and i1 of the tile's slot rows (equal when they share
            // one); columns past N read row 0 and store nothing.
            const int n_first = tl.n0 + col0;
            const int n_last = min(n_first + COLS, p.N) - 1;
            const int fb = tl.n0 / 128;
            int i0 = n_first < p.N ? n_first / 128 - fb : 0;
            int i1 = n_first < p.N ? n_last / 128 - fb : 0;
            if (SWIGLU) {                   // slot rows: 0 = w1's block, 1 = w3's
                i0 = 0;
                i1 = 1;
            }
            uint32_t upper = 0;             // bit c: slice c lies in block i1
#pragma unroll
            for (int c = 0; c < NCH; ++c)
                if (SWIGLU ? c >= NCH / 2 : (n_first < p.N && (n_first + SW * c) / 128 - fb != i0)) upper |= 1u << c;
            const int nk = tl.kb1 - tl.kb0;

            // running sums as packed fp32 pairs: acc[j] = (column 2j, column 2j+1)
            uint64_t acc[COLS / 2];
#pragma unroll
            for (int i = 0; i < COLS / 2; ++i) acc[i] = 0;

            for (int j = 0; j < nk; ++j, ++it) {
                const int b = it % NBUF;
                const uint32_t bph = (it / NBUF) & 1u;
                const int kb = tl.kb0 + j;
                const int c4 = kb % kScaleChunks;
                const int sl = ss % kScaleSlots;
                if ((j == 0 || c4 == 0) && !warp_wait(sfull_bar(sl), (ss / kScaleSlots) & 1u, ctl)) {
                    ok = false;
                    break;
                }
                if (j == 0 && p.bias != nullptr) {
                    // fused bias: the sums start from the bias (any fp32 summation
                    // order is within the result's bound)
                    const uint16_t* bias_s =
                        reinterpret_cast<const uint16_t*>(smem + L::OFF_BIAS + sl * L::BIAS_SLOT) + col0;
#pragma unroll
                    for (int v = 0; v < COLS / 8; ++v) {
                        const uint4 b8 = *reinterpret_cast<const uint4*>(bias_s + 8 * v);
                        const uint32_t bw[4] = {b8.x, b8.y, b8.z, b8.w};
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            acc[4 * v + t] = pack_f32x2(__uint_as_float(bw[t] << 16), __uint_as_float(bw[t] & 0xFFFF0000u));
                    }
                }
                if constexpr (MODE == kWgrad) {
                    // acc += RN(a * b_col) * P per element: a = sdy[chunk][n] of this
                    // thread's row, b_col = sx[chunk][k] of each column (slot layout
                    // [chunk][row] and [chunk][column]).  The column factors are
                    // read after the TMEM load, so the slot is freed afterwards.
                    const float a = sx_slots[sl * (BM * kScaleChunks) + c4 * BM + row];
                    if (!warp_wait(tfull_bar(b), bph, ctl)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t taddr = tmem + t_lane + static_cast<uint32_t>(b * L::BUF_COLS + col0);
                    static_assert(MODE != kWgrad || WHOLE, "weight-gradient tiles load a whole chunk at once");
                    uint64_t pr[COLS / 2];
                    tmem_ld_cols_pairs(taddr, pr);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty_bar(b));
                    const uint4* cf = reinterpret_cast<const uint4*>(
                        reinterpret_cast<const float*>(smem + L::OFF_CF + sl * L::CF_SLOT) + c4 * BN + col0);
                    const uint64_t a2 = pack_f32x2(a, a);
#pragma unroll
                    for (int v = 0; v < COLS / 4; ++v) {
                        const uint4 b4 = cf[v];
                        const uint64_t b01 = (static_cast<uint64_t>(b4.y) << 32) | b4.x;
                        const uint64_t b23 = (static_cast<uint64_t>(b4.w) << 32) | b4.z;
                        acc[2 * v] = f2_fma(f2_mul(a2, b01), pr[2 * v], acc[2 * v]);
                        acc[2 * v + 1] = f2_fma(f2_mul(a2, b23), pr[2 * v + 1], acc[2 * v + 1]);
                    }
                    if (c4 == kScaleChunks - 1 || j == nk - 1) {  // the block's last chunk here: free the slot
                        __syncwarp();
                        if (lane == 0) mbar_arrive(sempty_bar(sl));
                        ++ss;
                    }
                    continue;
                }
                const float* swv = sw_slots + sl * (kSwBlocks * kScaleChunks) + c4;
                const float sxv = sx_slots[sl * (BM * kScaleChunks) + row * kScaleChunks + c4];
                const float f_lo = __fmul_rn(sxv, swv[i0 * kScaleChunks]);
                const float f_hi = __fmul_rn(sxv, swv[i1 * kScaleChunks]);
                if (c4 == kScaleChunks - 1 || j == nk - 1) {  // the block's last chunk here: free the slot
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sempty_bar(sl));
                    ++ss;
                }
                const uint64_t f2lo = pack_f32x2(f_lo, f_lo), f2hi = pack_f32x2(f_hi, f_hi);
                uint64_t f2[NF];  // fp32(sx * sw) of each slice, as a packed pair
#pragma unroll
                for (int c = 0; c < NF; ++c) f2[c] = SWIGLU ? (c ? f2hi : f2lo) : ((upper >> c) & 1u) ? f2hi : f2lo;
                if (!warp_wait(tfull_bar(b), bph, ctl)) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = tmem + t_lane + static_cast<uint32_t>(b * L::BUF_COLS + col0);
                // promotion: acc += f * P_kb
                if constexpr (WHOLE) {
                    uint64_t pr[COLS / 2];
                    tmem_ld_cols_pairs(taddr, pr);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty_bar(b));  // the MMA may refill this buffer now
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
                        fma_pairs(*reinterpret_cast<uint64_t(*)[SP]>(&acc[SP * c]),
                                  *reinterpret_cast<uint64_t(*)[SP]>(&pr[SP * c]), f2[fsel(c)]);
                    continue;
                }
                uint64_t bufA[SP], bufB[SP];  // slices alternate between two buffers
                tmem_ld_x16_pairs(taddr, bufA);
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    uint64_t(&a)[SP] = *reinterpret_cast<uint64_t(*)[SP]>(&acc[SP * c]);
                    uint64_t(&cur)[SP] = (c & 1) ? bufB : bufA;
                    uint64_t(&nxt)[SP] = (c & 1) ? bufA : bufB;
                    const uint64_t fc = f2[fsel(c)];
                    if (c + 1 < NCH) {
                        tmem_ld_x16_pairs_fma(taddr + slice_col(c + 1), nxt, a, cur, fc);
                    } else {
                        fma_pairs(a, cur, fc);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(b));
            }
            if (!ok) break;
            const int nbase = tl.n0 + col0;
            if constexpr (SWIGLU) {
                // h = silu(gate) * up over the warpgroup's 64 columns, with the
                // bf16 roundings of the expert forward on bf16 tensors: each
                // GEMM output, silu (computed in fp32), and the product
                uint32_t hw[32];
#pragma unroll
                for (int v = 0; v < 32; ++v) {
                    float hv[2];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float g = bf16_round(j ? hi_f32(acc[v]) : lo_f32(acc[v]));
                        const float u = bf16_round(j ? hi_f32(acc[32 + v]) : lo_f32(acc[32 + v]));
                        const float sg = bf16_round(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))));
                        hv[j] = __fmul_rn(sg, u);
                    }
                    hw[v] = pack_bf16x2(hv[0], hv[1]);
                }
                GroupScale gs{};
                bool zero = true;
                if (p.yq != nullptr) {
                    // FP8 h: a row's 128-column group is split between the two
                    // warpgroups (64 columns each).  Each warp posts its rows'
                    // amax, arrives once on the tile parity's barrier (all
                    // lanes take part, before rows past the expert drop out)
                    // and reads the other warpgroup's after a bounded wait.
                    uint32_t amax2 = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        amax2 = absmax_bits8(make_uint4(hw[4 * i], hw[4 * i + 1], hw[4 * i + 2], hw[4 * i + 3]), amax2);
                    const float amax_own = bits_to_amax(amax2);
                    const uint32_t par = h_tiles & 1u;
                    float* hamax = reinterpret_cast<float*>(smem + L::OFF_HAMAX) + par * (2 * BM);
                    hamax[wg * BM + row] = amax_own;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(h_bar(par));
                    if (!warp_wait(h_bar(par), (h_tiles >> 1) & 1u, ctl)) { ok = false; break; }
                    ++h_tiles;
                    const float amax = fmaxf(amax_own, hamax[(1 - wg) * BM + row]);
                    gs = group_scale(amax);
                    zero = amax == 0.0f;
                }
                if (!row_ok) continue;
                if (p.yq != nullptr) {
                    uint8_t* qr = p.yq + static_cast<int64_t>(m) * p.ldyq + nbase;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint2 c0 = encode8(make_uint4(hw[8 * i], hw[8 * i + 1], hw[8 * i + 2], hw[8 * i + 3]), gs, zero);
                        const uint2 c1 = encode8(make_uint4(hw[8 * i + 4], hw[8 * i + 5], hw[8 * i + 6], hw[8 * i + 7]), gs, zero);
                        *reinterpret_cast<uint4*>(qr + 16 * i) = make_uint4(c0.x, c0.y, c1.x, c1.y);
                    }
                    if (wg == 0) p.sy[static_cast<int64_t>(m) * p.ldsy + tl.n0 / 128] = gs.s;
                }
                if (p.y != nullptr) {
                    uint16_t* hr = p.y + static_cast<int64_t>(m) * p.ldy + nbase;
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        *reinterpret_cast<uint4*>(hr + 8 * v) =
                            make_uint4(hw[4 * v], hw[4 * v + 1], hw[4 * v + 2], hw[4 * v + 3]);
                }
                continue;
            }
            if constexpr (MODE == kWgrad) {
                if (!row_ok) continue;
                float* yr = p.yf + static_cast<int64_t>(m) * p.ldyf;
#pragma unroll
                for (int v = 0; v < COLS / 4; ++v) {
                    const int n = nbase + 4 * v;
                    const float q[4] = {lo_f32(acc[2 * v]), hi_f32(acc[2 * v]), lo_f32(acc[2 * v + 1]),
                                        hi_f32(acc[2 * v + 1])};
                    if (n + 4 <= p.N) {
                        *reinterpret_cast<float4*>(yr + n) = make_float4(q[0], q[1], q[2], q[3]);
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            if (n + jj < p.N) yr[n + jj] = q[jj];
                    }
                }
                continue;
            }
            if (MODE == kSplitK) {
                if (!row_ok) continue;
                float* pr = p.partial + (static_cast<int64_t>(tl.tile) * p.M + m) * p.N;
#pragma unroll
                for (int v = 0; v < COLS / 4; ++v) {
                    const int n = nbase + 4 * v;
                    const float q[4] = {lo_f32(acc[2 * v]), hi_f32(acc[2 * v]), lo_f32(acc[2 * v + 1]),
                                        hi_f32(acc[2 * v + 1])};
                    if (n + 4 <= p.N && (p.N & 3) == 0) {
                        *reinterpret_cast<float4*>(pr + n) = make_float4(q[0], q[1], q[2], q[3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (n + j < p.N) pr[n + j] = q[j];
                    }
                }
            } else {
                uint32_t yb[COLS / 2];  // bf16 pairs (column 2v in the low half)
#pragma unroll
                for (int v = 0; v < COLS / 2; ++v) yb[v] = pack_bf16x2(lo_f32(acc[v]), hi_f32(acc[v]));
                // Whole 32-row boxes go out through shared memory: the warp's
                // 32 rows x 16 columns at a time, alternating between its two
                // 1 KB boxes (32-byte swizzle: the 16-byte half c of row r sits
                // at r * 32 + 16 * (c ^ ((r >> 2) & 1)), so the warp's stores
                // hit distinct banks), one TMA store per box.
                bool direct = p.y != nullptr;
                if constexpr (TMA_EPI) {
                    const int r0 = tl.m0 + quarter * 32;
                    if (p.y != nullptr && (MODE == kDense || r0 + 32 <= tl.m_end)) {
                        direct = false;
                        const uint32_t stage = sbase + L::OFF_EPI + static_cast<uint32_t>(ew) * 2048u;
                        const bool rows_in = r0 < p.M;
#pragma unroll
                        for (int pc = 0; pc < COLS / 16; ++pc, ++epi_n) {
                            const uint32_t box = stage + (epi_n & 1u) * 1024u;
                            if (lane == 0) bulk_wait_group_read<1>();  // the store two boxes back has read it
                            __syncwarp();
#pragma unroll
                            for (int c = 0; c < 2; ++c) {
                                const uint32_t dst = box + lane * 32 + 16 * (c ^ ((lane >> 2) & 1));
                                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst),
                                             "r"(yb[8 * pc + 4 * c]), "r"(yb[8 * pc + 4 * c + 1]),
                                             "r"(yb[8 * pc + 4 * c + 2]), "r"(yb[8 * pc + 4 * c + 3])
                                             : "memory");
                            }
                            fence_proxy_async_shared();
                            __syncwarp();
                            if (lane == 0) {
                                // a box wholly outside y is not stored, but its
                                // (empty) group is still committed: the buffer
                                // reuse above counts one group per box
                                if (rows_in && nbase + 16 * pc < p.N) tma_store_2d(&tmY, box, nbase + 16 * pc, r0);
                                bulk_commit_group();
                            }
                        }
                    }
                }
                if (!row_ok) continue;
                if (direct) {
                    uint16_t* yr = p.y + static_cast<int64_t>(m) * p.ldy;
#pragma unroll
                    for (int v = 0; v < COLS / 8; ++v) {
                        const int n = nbase + 8 * v;
                        if (n + 8 <= p.N) {
                            *reinterpret_cast<uint4*>(yr + n) =
                                make_uint4(yb[4 * v], yb[4 * v + 1], yb[4 * v + 2], yb[4 * v + 3]);
                        } else if (n < p.N) {
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                if (n + j < p.N) yr[n + j] = static_cast<uint16_t>(yb[4 * v + j / 2] >> (16 * (j & 1)));
                        }
                    }
                }
                if constexpr (COLS == 128 && BN % 128 == 0 && !SWIGLU) {
                    // The warpgroup's 128 columns are exactly one output group
                    // (the host asks for yq only with N % 128 == 0).
                    if (p.yq != nullptr && nbase < p.N) {
                        uint32_t amax2 = 0;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            amax2 = absmax_bits8(make_uint4(yb[4 * i], yb[4 * i + 1], yb[4 * i + 2], yb[4 * i + 3]),
                                                 amax2);
                        const float amax = bits_to_amax(amax2);
                        const GroupScale gs = group_scale(amax);
                        const bool zero = amax == 0.0f;
                        uint8_t* qr = p.yq + static_cast<int64_t>(m) * p.ldyq + nbase;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint2 c0 = encode8(
                                make_uint4(yb[8 * i], yb[8 * i + 1], yb[8 * i + 2], yb[8 * i + 3]), gs, zero);
                            const uint2 c1 = encode8(
                                make_uint4(yb[8 * i + 4], yb[8 * i + 5], yb[8 * i + 6], yb[8 * i + 7]), gs, zero);
                            *reinterpret_cast<uint4*>(qr + 16 * i) = make_uint4(c0.x, c0.y, c1.x, c1.y);
                        }
                        p.sy[static_cast<int64_t>(m) * p.ldsy + nbase / 128] = gs.s;
                    }
                }
            }
        }
        if constexpr (TMA_EPI) {  // the output boxes must be written before the CTA exits
            if (lane == 0) bulk_wait_group<0>();
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// Deterministic split-K reduction: y = bf16(sum over splits in order 0..S-1).
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ part, int splits, int M,
                                                           int N, uint16_t* __restrict__ y, int64_t ldy) {
    grid_dependency_wait();  // the partial sums come from the GEMM just before
    allow_dependents();
    const int64_t nch = (N + 7) / 8;
    const int64_t total = static_cast<int64_t>(M) * nch;
    const bool vec = (N & 3) == 0;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = idx / nch;
        const int n = static_cast<int>(idx - m * nch) * 8;
        float s[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j] = 0.0f;
        for (int sp = 0; sp < splits; ++sp) {
            const float* src = part + (static_cast<int64_t>(sp) * M + m) * N + n;
            if (vec && n + 8 <= N) {
                const float4 a = __ldg(reinterpret_cast<const float4*>(src));
                const float4 b = __ldg(reinterpret_cast<const float4*>(src + 4));
                s[0] += a.x; s[1] += a.y; s[2] += a.z; s[3] += a.w;
                s[4] += b.x; s[5] += b.y; s[6] += b.z; s[7] += b.w;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (n + j < N) s[j] += src[j];
            }
        }
        uint16_t* dst = y + m * ldy + n;
        if (n + 8 <= N) {
            uint4 o;
            o.x = pack_bf16x2(s[0], s[1]);
            o.y = pack_bf16x2(s[2], s[3]);
            o.z = pack_bf16x2(s[4], s[5]);
            o.w = pack_bf16x2(s[6], s[7]);
            *reinterpret_cast<uint4*>(dst) = o;
        } else {
            for (int j = 0; j < 8; ++j)
                if (n + j < N) {
                    const __nv_bfloat16 h = __float2bfloat16_rn(s[j]);
                    dst[j] = *reinterpret_cast<const uint16_t*>(&h);
                }
        }
    }
}

// ------------------------------------------------------------------ host side

// 2-D uint8 tensor [rows, inner] with the given row stride, boxes of
// box_rows x 128 bytes, 128-byte swizzle, zero fill outside the tensor.
cudaError_t make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t stride_bytes,
                     uint32_t box_rows) {
    return make_tmap_2d(map, base, 1, inner, rows, stride_bytes, BK, box_rows, 128);
}

// Tile widths 256, 192 or 160 columns.  A CTA's time per 128-K chunk is set
// by the round trip of its TMEM buffers (MMA, promotion, release) more than
// by the MMA width.  Measured on B300, relative to 256-column tiles (two TMEM
// buffers, two promotion warpgroups of 128 columns): 192-column tiles with
// three promotion warpgroups 0.91, 160-column tiles (three buffers) 0.77.
// The width with the fewest waves of tiles times that period wins; ties go to
// the wider tile.  (144-column tiles, 0.81, never need fewer waves than 160;
// 128-column tiles measured slower everywhere.)  Stages: as many 128-K
// stages as fit in shared memory next to the tables and the scale slots.
constexpr int kStages256 = 4;  // (16 + 32) KB per stage
constexpr int kStages160 = 5;  // (16 + 20) KB per stage
constexpr int kStages192 = 5;  // (16 + 24) KB per stage

int pick_bn(int64_t M, int64_t N, int num_sms) {
    constexpr int kWidths[3] = {256, 192, 160};
    constexpr int kPeriod[3] = {100, 91, 77};  // relative chunk period
    int best = 256;
    int64_t best_cost = INT64_MAX;
    for (int i = 0; i < 3; ++i) {
        const int64_t tiles = ((M + BM - 1) / BM) * ((N + kWidths[i] - 1) / kWidths[i]);
        const int64_t cost = ((tiles + num_sms - 1) / num_sms) * kPeriod[i];
        if (cost < best_cost) {
            best_cost = cost;
            best = kWidths[i];
        }
    }
    return best;
}

struct Plan {
    int bn;
    int mode;      // kDense or kSplitK
    int grid;
    int splits, kps;
    int64_t tiles;
    size_t ws;     // workspace bytes the plan uses
};

// Split-K when the tiles occupy less than half of the SMs (small M): each
// tile's 128-K chunks are cut into up to num_sms / tiles ranges of at least
// two chunks, the partial sums go to the workspace, and a second kernel adds
// them in split order.  Such shapes fit one wave at either width, so they
// always take the 160-column tiles.  Otherwise one CTA per tile (persistent).
Plan dense_plan(int64_t M, int64_t N, int64_t K, int num_sms, size_t ws_cap) {
    Plan pl{};
    pl.bn = pick_bn(M, N, num_sms);
    const int64_t KB = K / 128;
    pl.tiles = ((M + BM - 1) / BM) * ((N + pl.bn - 1) / pl.bn);
    pl.mode = kDense;
    pl.splits = 1;
    pl.kps = static_cast<int>(KB);
    pl.grid = static_cast<int>(std::min<int64_t>(pl.tiles, num_sms));
    pl.ws = 0;
    if (pl.tiles * 2 > num_sms || KB < 4) return pl;
    if (pl.bn != 160) return pl;  // not reached with the widths above; split-K is built for 160 only
    for (int64_t splits = std::min<int64_t>(num_sms / pl.tiles, KB / 2); splits > 1; --splits) {
        const int64_t kps = (KB + splits - 1) / splits;
        const int64_t s = (KB + kps - 1) / kps;
        const size_t ws = static_cast<size_t>(s) * static_cast<size_t>(M) * static_cast<size_t>(N) * sizeof(float);
        if (ws <= ws_cap) {
            pl.mode = kSplitK;
            pl.splits = static_cast<int>(s);
            pl.kps = static_cast<int>(kps);
            pl.grid = static_cast<int>(std::min<int64_t>(pl.tiles * s, num_sms));
            pl.ws = ws;
            return pl;
        }
    }
    return pl;
}

template <int BN, int STAGES, int MODE>
cudaError_t ensure_kernel_ready(int device) {
    static std::mutex mu;
    static bool done[64];
    std::lock_guard<std::mutex> g(mu);
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (!done[device]) {
        auto* k = fp8_gemm_kernel<BN, STAGES, MODE>;
        // The setmaxnreg split assumes exactly Roles::kRegsLaunch registers per
        // thread at launch; any other count could leave a warpgroup waiting
        // for registers that never free up.
        cudaError_t e;
        cudaFuncAttributes attr;
        if ((e = cudaFuncGetAttributes(&attr, k)) != cudaSuccess) return e;
        if (attr.numRegs != Roles<nwg_for(BN)>::kRegsLaunch) return cudaErrorInvalidKernelImage;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<BN, STAGES>::ALLOC);
        if (e != cudaSuccess) return e;
        done[device] = true;
    }
    return cudaSuccess;
}

template <int BN, int STAGES, int MODE>
cudaError_t launch_mode(const GemmArgs& a, Params& p, int grid, const DeviceInfo& dev, cudaStream_t stream) {
    const int64_t b_rows = is_grouped(MODE) ? static_cast<int64_t>(a.G) * a.N : a.N;
    CUtensorMap tmA, tmB, tmB3, tmS, tmY;
    cudaError_t e;
    if ((e = make_map(&tmA, a.xq, a.K, a.M, a.K, BM)) != cudaSuccess) return e;
    if constexpr (MODE == kGroupedSwiglu) {  // two boxes of 128 rows per stage, one from each weight
        if ((e = make_map(&tmB, a.wq, a.K, b_rows, a.K, 128)) != cudaSuccess) return e;
        if ((e = make_map(&tmB3, a.wq3, a.K, b_rows, a.K, 128)) != cudaSuccess) return e;
    } else {
        if ((e = make_map(&tmB, a.wq, a.K, b_rows, a.K, BN)) != cudaSuccess) return e;
        tmB3 = tmB;  // unused
    }
    // sx [M, lds] fp32: boxes of kScaleChunks chunks x BM rows
    if ((e = make_tmap_2d(&tmS, a.sx, 4, a.lds, a.M, a.lds * 4, kScaleChunks, BM, 0)) != cudaSuccess) return e;
    // y [M, N] bf16 with row stride ldy: boxes of 32 rows x 16 columns for
    // the TMA-store epilogue of 256-column dense / grouped tiles
    if (BN == 256 && (MODE == kDense || MODE == kGrouped) && a.y != nullptr) {
        if ((e = make_tmap_2d(&tmY, a.y, 2, a.N, a.M, a.ldy * 2, 16, 32, 32)) != cudaSuccess) return e;
    } else {
        tmY = tmA;  // unused
    }
    if ((e = ensure_kernel_ready<BN, STAGES, MODE>(dev.device)) != cudaSuccess) return e;
    return launch_pdl(fp8_gemm_kernel<BN, STAGES, MODE>, dim3(grid), dim3(Roles<nwg_for(BN)>::kThreads),
                      Layout<BN, STAGES>::ALLOC,
                      stream, tmA, tmB, tmB3, tmS, tmY, p);
}

template <int MODE>
cudaError_t launch_bn(int bn, const GemmArgs& a, Params& p, int grid, const DeviceInfo& dev, cudaStream_t stream) {
    if (bn == 160) return launch_mode<160, kStages160, MODE>(a, p, grid, dev, stream);
    if constexpr (MODE == kSplitK) {
        return cudaErrorNotSupported;  // split-K plans use 160 only
    } else {
        if (bn == 192) return launch_mode<192, kStages192, MODE>(a, p, grid, dev, stream);
        return launch_mode<256, kStages256, MODE>(a, p, grid, dev, stream);
    }
}

}  // namespace

size_t gemm_workspace_size(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev) {
    if (gemm_skinny_applies(M, N, K)) return 0;
    return dense_plan(M, N, K, dev.num_sms, ~size_t{0}).ws;
}

cudaError_t launch_gemm(const GemmArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
    Params p{};
    p.sx = a.sx;
    p.lds = a.lds;
    p.sw = a.sw;
    p.y = a.y;
    p.ldy = a.ldy;
    p.M = static_cast<int>(a.M);
    p.N = static_cast<int>(a.N);
    p.KB = static_cast<int>(a.K / 128);
    p.err = dev.err;
    p.timeout_ns = wait_timeout_ns();
    if (a.offsets != nullptr) {
        p.offsets = a.offsets;
        p.G = a.G;
        if (a.wq3 != nullptr) {
            p.sw3 = a.sw3;
            p.yq = a.yq;
            p.ldyq = a.ldyq;
            p.sy = a.sy;
            p.ldsy = a.ldsy;
            return launch_mode<256, kStages256, kGroupedSwiglu>(a, p, dev.num_sms, dev, stream);
        }
        return launch_mode<256, kStages256, kGrouped>(a, p, dev.num_sms, dev, stream);
    }
    const bool fused = a.bias != nullptr || a.yq != nullptr;
    if (!fused && gemm_skinny_applies(a.M, a.N, a.K)) return launch_gemm_skinny(a, dev, stream);
    Plan pl = dense_plan(a.M, a.N, a.K, dev.num_sms, a.workspace && !fused ? a.ws_bytes : 0);
    if (a.yq != nullptr && pl.bn != 256) {
        // Output quantisation needs each promotion warpgroup to hold one whole
        // 128-column group: 256-column tiles, whatever the cost model prefers.
        pl.bn = 256;
        pl.tiles = ((a.M + BM - 1) / BM) * ((a.N + 255) / 256);
        pl.grid = static_cast<int>(std::min<int64_t>(pl.tiles, dev.num_sms));
    }
    p.bias = a.bias;
    p.yq = a.yq;
    p.ldyq = a.ldyq;
    p.sy = a.sy;
    p.ldsy = a.ldsy;
    p.MT = static_cast<int>((a.M + BM - 1) / BM);
    p.NT = static_cast<int>((a.N + pl.bn - 1) / pl.bn);
    p.splits = pl.splits;
    p.kps = pl.kps;
    p.num_tiles = static_cast<int>(pl.tiles * pl.splits);
    cudaError_t e;
    if (pl.mode == kSplitK) {
        p.partial = static_cast<float*>(a.workspace);
        e = launch_bn<kSplitK>(pl.bn, a, p, pl.grid, dev, stream);
        if (e != cudaSuccess) return e;
        const int64_t work = a.M * ((a.N + 7) / 8);
        const int blocks = static_cast<int>(std::min<int64_t>((work + 255) / 256, dev.num_sms * 8));
        return launch_pdl(splitk_reduce_kernel, dim3(blocks), dim3(256), 0, stream,
                          static_cast<const float*>(p.partial), pl.splits, p.M, p.N, a.y, a.ldy);
    }
    return launch_bn<kDense>(pl.bn, a, p, pl.grid, dev, stream);
}

cudaError_t launch_wgrad(const WgradArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
    constexpr int BN = 160;
    const int64_t TB = (a.T + 127) / 128;
    Params p{};
    p.M = static_cast<int>(a.N);
    p.N = static_cast<int>(a.K);
    p.KB = static_cast<int>(TB);
    p.MT = static_cast<int>((a.N + BM - 1) / BM);
    p.NT = static_cast<int>((a.K + BN - 1) / BN);
    p.num_tiles = p.MT * p.NT;
    p.yf = a.dw;
    p.ldyf = a.lddw;
    p.err = dev.err;
    p.timeout_ns = wait_timeout_ns();
    CUtensorMap tmA, tmB, tmS, tmC;
    cudaError_t e;
    // operands: rows of dY^T and X^T, tokens contiguous (128-token K chunks)
    if ((e = make_map(&tmA, a.dyqt, a.T, a.N, a.lddyt, BM)) != cudaSuccess) return e;
    if ((e = make_map(&tmB, a.xqt, a.T, a.K, a.ldxt, BN)) != cudaSuccess) return e;
    // row factors sdy [TB, N] and column factors sx [TB, K]: boxes of one
    // tile's rows (columns) for kScaleChunks token chunks
    if ((e = make_tmap_2d(&tmS, a.sdy, 4, a.N, TB, a.ldsdy * 4, BM, kScaleChunks, 0)) != cudaSuccess) return e;
    if ((e = make_tmap_2d(&tmC, a.sx, 4, a.K, TB, a.ldsx * 4, BN, kScaleChunks, 0)) != cudaSuccess) return e;
    if ((e = ensure_kernel_ready<BN, kStages160, kWgrad>(dev.device)) != cudaSuccess) return e;
    const int grid = std::min(p.num_tiles, dev.num_sms);
    return launch_pdl(fp8_gemm_kernel<BN, kStages160, kWgrad>, dim3(grid), dim3(Roles<nwg_for(BN)>::kThreads),
                      Layout<BN, kStages160>::ALLOC, stream, tmA, tmB, tmC, tmS, tmA, p);
}

}  // namespace fp8bs
