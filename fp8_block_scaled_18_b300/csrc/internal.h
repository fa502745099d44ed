// internal.h -- launchers shared between the C-ABI shim (api.cu) and the
// kernel translation units.  Arguments are validated by the shim before any
// launcher runs.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fp8bs {

// Status-word bit set by the MoE gathers when a routed row or token id lies
// outside its range (the wait-timeout bits, 1 and 2, are defined with the
// bounded waits in ptx.cuh).
constexpr unsigned kDevErrIndex = 4u;

struct DeviceInfo {
    int device;
    int num_sms;
    unsigned* err;  // device address of this device's status word
};

// Per-device facts, filled once per device under a lock (status.cu).
cudaError_t device_info(DeviceInfo* out);

// Nanoseconds a pipeline wait may take before the kernel gives up
// (FP8BS_WAIT_TIMEOUT_NS in the environment overrides the default of 2 s).
uint64_t wait_timeout_ns();

// Encode a 2-D TMA descriptor over a row-major tensor [rows, inner] of
// elem_bytes-sized elements (1, 2 or 4; 4 = fp32) with the given row stride in bytes;
// boxes of box_rows x box_inner elements; swizzle_bytes 128, 64 or 32 selects
// that shared-memory swizzle (128: the MMA operand layout), 0 none.  Loads
// outside the tensor fill with zeros; stores outside it are dropped.
// (tmap.cu)
cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner, uint64_t rows,
                         uint64_t stride_bytes, uint32_t box_inner, uint32_t box_rows, int swizzle_bytes);

// Launch `kernel` with programmatic stream serialisation: it may begin while
// the previous kernel in `stream` finishes; the kernel itself waits
// (grid_dependency_wait) before touching global memory.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// pow2: power-of-two (UE8M0-style) scales rounded up instead of amax / 448.
cudaError_t launch_act_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq, int64_t ldq,
                             float* sx, int64_t lds, const DeviceInfo& dev, cudaStream_t stream, bool pow2 = false);
cudaError_t launch_weight_quant(const uint16_t* w, int64_t N, int64_t K, uint8_t* wq, float* sw,
                                const DeviceInfo& dev, cudaStream_t stream, bool pow2 = false);
cudaError_t launch_weight_dequant(const uint8_t* wq, const float* sw, int64_t N, int64_t K, uint16_t* w,
                                  const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_e4m3_encode(const float* v, int64_t n, uint8_t* q, const DeviceInfo& dev,
                               cudaStream_t stream);
cudaError_t launch_wait_selftest(uint64_t timeout_ns, const DeviceInfo& dev, cudaStream_t stream);

// MoE dispatch and combine (moe.cu).
cudaError_t launch_moe_dispatch(const uint8_t* xq, int64_t ldq, const float* sx, int64_t lds, int64_t tokens,
                                int64_t K, const int32_t* token_of_row, int64_t R, uint8_t* xr, int64_t ldr,
                                float* sr, int64_t ldsr, const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_moe_combine(const uint16_t* yk, int64_t ldyk, int64_t R, const float* w,
                               const int32_t* rows_of_token, int64_t tokens, int32_t topk, int64_t dim,
                               const uint16_t* z, int64_t ldz, uint16_t* y, int64_t ldy, const DeviceInfo& dev,
                               cudaStream_t stream);

// MoE router (router.cu).
cudaError_t launch_moe_gate(const uint16_t* x, int64_t ldx, const uint16_t* wg, const float* bias, int64_t T,
                            int64_t dim, int E, int n_groups, int topk_groups, int top_k, float route_scale,
                            int32_t* ids, float* w, const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_moe_route(const int32_t* ids, const float* w, int64_t T, int top_k, int E, int32_t* offsets,
                             int32_t* token_of_row, int32_t* rows_of_token, float* weight_of_row,
                             const DeviceInfo& dev, cudaStream_t stream);

// Dense and grouped GEMM (gemm.cu).
struct GemmArgs {
    const uint8_t* xq;
    const float* sx;
    int64_t lds;
    const uint8_t* wq;
    const float* sw;
    int64_t M, N, K;
    uint16_t* y;
    int64_t ldy;
    // grouped only
    const int32_t* offsets;  // device [G+1] or nullptr for a dense GEMM
    int32_t G;
    // dense split-K scratch
    void* workspace;
    size_t ws_bytes;
    // fused epilogue (dense only; no split-K): bias bf16 [N] or nullptr; yq
    // e4m3 [M, ldyq] + sy fp32 [M, ldsy] or nullptr (then N % 128 == 0)
    // SwiGLU grouped (then y = h [M, ldy], N = the intermediate size): w3's
    // operand and scales, laid out like wq / sw
    const uint8_t* wq3 = nullptr;
    const float* sw3 = nullptr;
    const uint16_t* bias = nullptr;
    uint8_t* yq = nullptr;
    int64_t ldyq = 0;
    float* sy = nullptr;
    int64_t ldsy = 0;
};

size_t gemm_workspace_size(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev);
cudaError_t launch_gemm(const GemmArgs& a, const DeviceInfo& dev, cudaStream_t stream);
// Few tokens (M <= 128, K within 8 CTAs' chunk budget: 8192 for M <= 64,
// 4096 for M <= 128): the weight-streaming kernel of skinny.cu (one launch,
// no workspace); launch_gemm takes it for plain dense GEMMs.
bool gemm_skinny_applies(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_skinny(const GemmArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// Weight gradient dW [N, K] fp32 = dY^T X over T tokens from the column-
// quantised (128x1 groups along the tokens) operands, stored transposed:
// dyqt [N, lddyt] and xqt [K, ldxt] e4m3 (row = one channel's T tokens),
// sdy [ceil(T/128), ldsdy] and sx [ceil(T/128), ldsx] fp32 (gemm.cu).
struct WgradArgs {
    const uint8_t* dyqt;
    int64_t lddyt;
    const float* sdy;
    int64_t ldsdy;
    const uint8_t* xqt;
    int64_t ldxt;
    const float* sx;
    int64_t ldsx;
    int64_t T, N, K;
    float* dw;
    int64_t lddw;
};
cudaError_t launch_wgrad(const WgradArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// 128x1 column quantisation: per column k and per block of 128 rows, amax,
// s = amax / 448 and the codes, written transposed: xqt[k, m] (quant.cu).
cudaError_t launch_act_quant_cols(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xqt, int64_t ldt,
                                  float* sc, int64_t ldsc, const DeviceInfo& dev, cudaStream_t stream);

}  // namespace fp8bs
