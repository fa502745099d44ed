// moe.cu -- the routed-expert data movement around the grouped GEMMs:
// dispatch (quantised token rows gathered into expert order) and combine
// (each token's expert outputs summed with its gate values).  Both are
// HBM-bound gathers; neither touches the tensor cores.
//
// Routing facts they follow: every token keeps all of its top-k experts, no
// token is dropped, and the expert outputs are weighted by the gate values
// (the sigmoid affinities), not by the bias-adjusted scores that only steer
// the selection (page 2 of the DeepSeek-V3 notes, section 2-2); the shared
// experts' output, which every token receives, is added to the routed sum
// (page 3, the DeepSeekMoE shared-expert paragraph).
#include <cuda_bf16.h>

#include "codec.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

__device__ __forceinline__ uint4 ld_nc_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_nc(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ------------------------------------------------------------------ dispatch
//
// One warp per routed row: the source token's K codes move as 16-byte
// chunks (lane-strided, so each warp instruction covers 512 contiguous
// bytes), then its K/128 scales.  A token is read by up to top-k warps; the
// quantised token matrix (tokens x K bytes) is small enough to stay in L2
// between them, so HBM sees it about once.
constexpr int kDispatchUnroll = 4;

__global__ void __launch_bounds__(256) moe_dispatch_kernel(const uint8_t* __restrict__ xq, int64_t ldq,
                                                          const float* __restrict__ sx, int64_t lds,
                                                          int64_t tokens, const int32_t* __restrict__ token_of_row,
                                                          int64_t R, int64_t C, int64_t KB,
                                                          uint8_t* __restrict__ xr, int64_t ldr,
                                                          float* __restrict__ sr, int64_t ldsr,
                                                          unsigned* __restrict__ err) {
    grid_dependency_wait();
    allow_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r = warp; r < R; r += nwarps) {
        const int64_t t = __ldg(token_of_row + r);
        const bool ok = t >= 0 && t < tokens;
        if (!ok && lane == 0) atomicOr(err, kDevErrIndex);
        const uint8_t* src = xq + (ok ? t : 0) * ldq;
        uint8_t* dst = xr + r * ldr;
        for (int64_t c0 = lane; c0 < C; c0 += 32 * kDispatchUnroll) {
            uint4 v[kDispatchUnroll];
#pragma unroll
            for (int j = 0; j < kDispatchUnroll; ++j) {
                const int64_t c = c0 + 32 * j;
                v[j] = (ok && c < C) ? ld_nc(src + c * 16) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < kDispatchUnroll; ++j) {
                const int64_t c = c0 + 32 * j;
                if (c < C) *reinterpret_cast<uint4*>(dst + c * 16) = v[j];
            }
        }
        for (int64_t kb = lane; kb < KB; kb += 32) sr[r * ldsr + kb] = ok ? __ldg(sx + t * lds + kb) : 0.0f;
    }
}

// ------------------------------------------------------------------- combine
//
// One thread per 8 consecutive outputs (16 bytes) of a token: it reads the
// token's routed row ids and their gate values (shared by the token's
// dim/8 threads, so they come from L1), issues the k expert-row loads of its
// 8 columns together (16 bytes each, streamed past L1: every expert output
// is read exactly once), and accumulates
//   acc = z;  acc = fma(w_k, yk_k, acc)  for k = 0 .. topk-1
// in fp32 (packed pairs, each one IEEE fused multiply-add), rounding once to
// bf16 at the end.  Consecutive threads take consecutive chunks of a row, so
// each warp's loads of one expert row are 512 contiguous bytes.
constexpr int kCombineBatch = 8;  // expert rows whose loads are in flight together

__global__ void __launch_bounds__(256) moe_combine_kernel(const uint16_t* __restrict__ yk, int64_t ldyk, int64_t R,
                                                         const float* __restrict__ w,
                                                         const int32_t* __restrict__ rows_of_token, int32_t topk,
                                                         const uint16_t* z, int64_t ldz, int64_t tokens, int64_t C,
                                                         uint16_t* y, int64_t ldy, unsigned* __restrict__ err) {
    grid_dependency_wait();
    allow_dependents();
    const int64_t total = tokens * C;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    bool bad = false;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t t = i / C;
        const int64_t c = i - t * C;
        uint64_t acc[4];
        if (z) {
            // plain load: z may be y itself (each thread reads its chunk before writing it)
            const uint4 v = *reinterpret_cast<const uint4*>(z + t * ldz + c * 8);
            acc[0] = f2(bf16_lo(v.x), bf16_hi(v.x));
            acc[1] = f2(bf16_lo(v.y), bf16_hi(v.y));
            acc[2] = f2(bf16_lo(v.z), bf16_hi(v.z));
            acc[3] = f2(bf16_lo(v.w), bf16_hi(v.w));
        } else {
            acc[0] = acc[1] = acc[2] = acc[3] = 0;
        }
        const int32_t* rt = rows_of_token + t * topk;
        for (int k0 = 0; k0 < topk; k0 += kCombineBatch) {
            uint4 v[kCombineBatch];
            float wk[kCombineBatch];
            unsigned use = 0;  // terms present: past topk, or with a row id out of range, are skipped
#pragma unroll
            for (int j = 0; j < kCombineBatch; ++j) {
                v[j] = make_uint4(0, 0, 0, 0);
                wk[j] = 0.0f;
                if (k0 + j < topk) {
                    const int64_t r = __ldg(rt + k0 + j);
                    if (r >= 0 && r < R) {
                        wk[j] = __ldg(w + r);
                        v[j] = ld_nc_stream(yk + r * ldyk + c * 8);
                        use |= 1u << j;
                    } else {
                        bad = true;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kCombineBatch; ++j) {
                if (use & (1u << j)) {
                    const uint64_t ww = f2(wk[j], wk[j]);
                    acc[0] = f2_fma(ww, f2(bf16_lo(v[j].x), bf16_hi(v[j].x)), acc[0]);
                    acc[1] = f2_fma(ww, f2(bf16_lo(v[j].y), bf16_hi(v[j].y)), acc[1]);
                    acc[2] = f2_fma(ww, f2(bf16_lo(v[j].z), bf16_hi(v[j].z)), acc[2]);
                    acc[3] = f2_fma(ww, f2(bf16_lo(v[j].w), bf16_hi(v[j].w)), acc[3]);
                }
            }
        }
        uint32_t out[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(static_cast<uint32_t>(acc[p])),
                                                           __uint_as_float(static_cast<uint32_t>(acc[p] >> 32)));
            out[p] = *reinterpret_cast<const uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(y + t * ldy + c * 8) = make_uint4(out[0], out[1], out[2], out[3]);
    }
    if (bad) atomicOr(err, kDevErrIndex);
}

template <typename Kernel>
int resident_blocks(Kernel k, int threads) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, 0) != cudaSuccess || n < 1) n = 1;
    return n;
}

}  // namespace

cudaError_t launch_moe_dispatch(const uint8_t* xq, int64_t ldq, const float* sx, int64_t lds, int64_t tokens,
                                int64_t K, const int32_t* token_of_row, int64_t R, uint8_t* xr, int64_t ldr,
                                float* sr, int64_t ldsr, const DeviceInfo& dev, cudaStream_t stream) {
    static const int per_sm = resident_blocks(moe_dispatch_kernel, 256);
    const int64_t blocks_needed = (R + 7) / 8;  // 8 warps per block, one row each
    const int64_t max_blocks = static_cast<int64_t>(dev.num_sms) * per_sm;
    const int blocks = static_cast<int>(blocks_needed < max_blocks ? blocks_needed : max_blocks);
    return launch_pdl(moe_dispatch_kernel, dim3(blocks), dim3(256), 0, stream, xq, ldq, sx, lds, tokens,
                      token_of_row, R, K / 16, K / 128, xr, ldr, sr, ldsr, dev.err);
}

cudaError_t launch_moe_combine(const uint16_t* yk, int64_t ldyk, int64_t R, const float* w,
                               const int32_t* rows_of_token, int64_t tokens, int32_t topk, int64_t dim,
                               const uint16_t* z, int64_t ldz, uint16_t* y, int64_t ldy, const DeviceInfo& dev,
                               cudaStream_t stream) {
    static const int per_sm = resident_blocks(moe_combine_kernel, 256);
    const int64_t C = dim / 8;
    const int64_t blocks_needed = (tokens * C + 255) / 256;
    const int64_t max_blocks = static_cast<int64_t>(dev.num_sms) * per_sm;
    const int blocks = static_cast<int>(blocks_needed < max_blocks ? blocks_needed : max_blocks);
    return launch_pdl(moe_combine_kernel, dim3(blocks), dim3(256), 0, stream, yk, ldyk, R, w, rows_of_token, topk,
                      z, ldz, tokens, C, y, ldy, dev.err);
}

}  // namespace fp8bs
