// api.cu -- the C ABI declared in include/fp8bs.h: argument validation, then
// one launch on the caller's stream.  Nothing here allocates device memory.
#include "../../include/fp8bs.h"
#include "internal.h"
#include "ptx.cuh"

using namespace fp8bs;

namespace {

constexpr int64_t kMaxRows = (int64_t{1} << 31) - 1;   // TMA coordinates are int32
constexpr int64_t kMaxGridY = 65535;
constexpr int32_t kMaxGroups = 1024;                    // grouped GEMM: per-CTA tile table

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline fp8bs_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FP8BS_OK : FP8BS_ERR_CUDA; }

inline fp8bs_status device(DeviceInfo* d) {
    if (device_info(d) != cudaSuccess) return FP8BS_ERR_CUDA;
    return FP8BS_OK;
}

inline cudaStream_t cs(fp8bs_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Shape checks common to the quantisers' K dimension.
inline fp8bs_status check_k(int64_t K) {
    if (K < 0) return FP8BS_ERR_INVALID_ARG;
    if (K == 0 || K % 128 != 0) return FP8BS_ERR_UNSUPPORTED;
    if (K / 128 > (int64_t{1} << 31) - 1) return FP8BS_ERR_UNSUPPORTED;
    return FP8BS_OK;
}

}  // namespace

extern "C" {

fp8bs_status fp8bs_act_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq, int64_t ldq,
                             float* sx, int64_t lds, fp8bs_stream_t stream) {
    if (M < 0) return FP8BS_ERR_INVALID_ARG;
    if (fp8bs_status st = check_k(K)) return st;
    if (M == 0) return FP8BS_OK;
    if (!x || !xq || !sx) return FP8BS_ERR_INVALID_ARG;
    if (ldx < K || ldq < K || lds < K / 128) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq) || !aligned16(sx) || ldx % 8 || ldq % 16 || lds % 4)
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    return from_cuda(launch_act_quant(x, M, K, ldx, xq, ldq, sx, lds, d, cs(stream)));
}

fp8bs_status fp8bs_weight_quant(const uint16_t* w, int64_t N, int64_t K, uint8_t* wq, float* sw,
                                fp8bs_stream_t stream) {
    if (N < 0) return FP8BS_ERR_INVALID_ARG;
    if (fp8bs_status st = check_k(K)) return st;
    if (N == 0) return FP8BS_OK;
    if (!w || !wq || !sw) return FP8BS_ERR_INVALID_ARG;
    if ((N + 127) / 128 > kMaxGridY) return FP8BS_ERR_UNSUPPORTED;
    if (!aligned16(w) || !aligned16(wq) || (reinterpret_cast<uintptr_t>(sw) & 3u)) return FP8BS_ERR_MISALIGNED;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    return from_cuda(launch_weight_quant(w, N, K, wq, sw, d, cs(stream)));
}

fp8bs_status fp8bs_act_quant_pow2(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq, int64_t ldq,
                                  float* sx, int64_t lds, fp8bs_stream_t stream) {
    if (M < 0) return FP8BS_ERR_INVALID_ARG;
    if (fp8bs_status st = check_k(K)) return st;
    if (M == 0) return FP8BS_OK;
    if (!x || !xq || !sx) return FP8BS_ERR_INVALID_ARG;
    if (ldx < K || ldq < K || lds < K / 128) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq) || !aligned16(sx) || ldx % 8 || ldq % 16 || lds % 4)
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    return from_cuda(launch_act_quant(x, M, K, ldx, xq, ldq, sx, lds, d, cs(stream), true));
}

fp8bs_status fp8bs_weight_quant_pow2(const uint16_t* w, int64_t N, int64_t K, uint8_t* wq, float* sw,
                                     fp8bs_stream_t stream) {
    if (N < 0) return FP8BS_ERR_INVALID_ARG;
    if (fp8bs_status st = check_k(K)) return st;
    if (N == 0) return FP8BS_OK;
    if (!w || !wq || !sw) return FP8BS_ERR_INVALID_ARG;
    if ((N + 127) / 128 > kMaxGridY) return FP8BS_ERR_UNSUPPORTED;
    if (!aligned16(w) || !aligned16(wq) || (reinterpret_cast<uintptr_t>(sw) & 3u)) return FP8BS_ERR_MISALIGNED;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    return from_cuda(launch_weight_quant(w, N, K, wq, sw, d, cs(stream), true));
}

fp8bs_status fp8bs_weight_dequant(const uint8_t* wq, const float* sw, int64_t N, int64_t K, uint16_t* w,
                                  fp8bs_stream_t stream) {
    if (N < 0) return FP8BS_ERR_INVALID_ARG;
    if (fp8bs_status st = check_k(K)) return st;
    if (N == 0) return FP8BS_OK;
    if (!w || !wq || !sw) return FP8BS_ERR_INVALID_ARG;
    if ((N + 127) / 128 > kMaxGridY) return FP8BS_ERR_UNSUPPORTED;
    if (!aligned16(w) || !aligned16(wq) || (reinterpret_cast<uintptr_t>(sw) & 3u)) return FP8BS_ERR_MISALIGNED;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    return from_cuda(launch_weight_dequant(wq, sw, N, K, w, d, cs(stream)));
}

static fp8bs_status check_gemm_common(const uint8_t* xq, const float* sx, int64_t lds, const uint8_t* wq,
                                      const float* sw, int64_t M, int64_t N, int64_t K, const uint16_t* y,
                                      int64_t ldy) {
    if (!xq || !sx || !wq || !sw || !y) return FP8BS_ERR_INVALID_ARG;
    if (M > kMaxRows || N > kMaxRows) return FP8BS_ERR_UNSUPPORTED;
    if (lds < K / 128 || ldy < N) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(xq) || !aligned16(wq) || !aligned16(sx) || !aligned16(y) || lds % 4 || ldy % 8 ||
        (reinterpret_cast<uintptr_t>(sw) & 3u))
        return FP8BS_ERR_MISALIGNED;
    return FP8BS_OK;
}

fp8bs_status fp8bs_gemm(const uint8_t* xq, const float* sx, int64_t lds, const uint8_t* wq, const float* sw,
                        int64_t M, int64_t N, int64_t K, uint16_t* y, int64_t ldy, void* workspace,
                        size_t ws_bytes, fp8bs_stream_t stream) {
    if (M < 0 || N < 0) return FP8BS_ERR_INVALID_ARG;
    if (fp8bs_status st = check_k(K)) return st;
    if (M == 0 || N == 0) return FP8BS_OK;
    if (fp8bs_status st = check_gemm_common(xq, sx, lds, wq, sw, M, N, K, y, ldy)) return st;
    if (workspace && !aligned16(workspace)) return FP8BS_ERR_MISALIGNED;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    GemmArgs a{xq, sx, lds, wq, sw, M, N, K, y, ldy, nullptr, 0, workspace, workspace ? ws_bytes : 0};
    return from_cuda(launch_gemm(a, d, cs(stream)));
}

fp8bs_status fp8bs_gemm_fused(const uint8_t* xq, const float* sx, int64_t lds, const uint8_t* wq, const float* sw,
                              const uint16_t* bias, int64_t M, int64_t N, int64_t K, uint16_t* y, int64_t ldy,
                              uint8_t* yq, int64_t ldyq, float* sy, int64_t ldsy, fp8bs_stream_t stream) {
    if (M < 0 || N < 0) return FP8BS_ERR_INVALID_ARG;
    if (fp8bs_status st = check_k(K)) return st;
    if (M == 0 || N == 0) return FP8BS_OK;
    if (!y && !yq) return FP8BS_ERR_INVALID_ARG;  // nothing to write
    if (!xq || !sx || !wq || !sw) return FP8BS_ERR_INVALID_ARG;
    if (M > kMaxRows || N > kMaxRows) return FP8BS_ERR_UNSUPPORTED;
    if (lds < K / 128) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(xq) || !aligned16(wq) || !aligned16(sx) || lds % 4 || (reinterpret_cast<uintptr_t>(sw) & 3u))
        return FP8BS_ERR_MISALIGNED;
    if (bias && (reinterpret_cast<uintptr_t>(bias) & 1u)) return FP8BS_ERR_MISALIGNED;
    if (y) {
        if (ldy < N) return FP8BS_ERR_INVALID_ARG;
        if (!aligned16(y) || ldy % 8) return FP8BS_ERR_MISALIGNED;
    }
    if (yq) {
        if (N % 128) return FP8BS_ERR_UNSUPPORTED;  // whole 128-column output groups only
        if (!sy) return FP8BS_ERR_INVALID_ARG;
        if (ldyq < N || ldsy < N / 128) return FP8BS_ERR_INVALID_ARG;
        if (!aligned16(yq) || ldyq % 16 || !aligned16(sy) || ldsy % 4) return FP8BS_ERR_MISALIGNED;
    }
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    GemmArgs a{xq, sx, lds, wq, sw, M, N, K, y, ldy, nullptr, 0, nullptr, 0};
    a.bias = bias;
    a.yq = yq;
    a.ldyq = ldyq;
    a.sy = sy;
    a.ldsy = ldsy;
    return from_cuda(launch_gemm(a, d, cs(stream)));
}

size_t fp8bs_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || K % 128) return 0;
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess) return 0;
    return gemm_workspace_size(M, N, K, d);
}

size_t fp8bs_grouped_gemm_workspace_size(int32_t, int64_t, int64_t) { return 0; }

fp8bs_status fp8bs_grouped_gemm(const uint8_t* xq, const float* sx, int64_t lds, const uint8_t* wq,
                                const float* sw, const int32_t* offsets_dev, int32_t G, int64_t total_M,
                                int64_t N, int64_t K, uint16_t* y, int64_t ldy, fp8bs_stream_t stream) {
    if (G < 0 || total_M < 0 || N < 0) return FP8BS_ERR_INVALID_ARG;
    if (fp8bs_status st = check_k(K)) return st;
    if (total_M == 0 || N == 0 || G == 0) return FP8BS_OK;
    if (!offsets_dev) return FP8BS_ERR_INVALID_ARG;
    if (G > kMaxGroups) return FP8BS_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(G) * N > kMaxRows) return FP8BS_ERR_UNSUPPORTED;
    if (fp8bs_status st = check_gemm_common(xq, sx, lds, wq, sw, total_M, N, K, y, ldy)) return st;
    if (reinterpret_cast<uintptr_t>(offsets_dev) & 3u) return FP8BS_ERR_MISALIGNED;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    GemmArgs a{xq, sx, lds, wq, sw, total_M, N, K, y, ldy, offsets_dev, G, nullptr, 0};
    return from_cuda(launch_gemm(a, d, cs(stream)));
}

fp8bs_status fp8bs_grouped_gemm_swiglu(const uint8_t* xq, const float* sx, int64_t lds, const uint8_t* w1q,
                                       const float* sw1, const uint8_t* w3q, const float* sw3,
                                       const int32_t* offsets_dev, int32_t G, int64_t total_M, int64_t I,
                                       int64_t K, uint16_t* h, int64_t ldh, uint8_t* hq, int64_t ldhq, float* sh,
                                       int64_t ldsh, fp8bs_stream_t stream) {
    if (G < 0 || total_M < 0 || I < 0) return FP8BS_ERR_INVALID_ARG;
    if (fp8bs_status st = check_k(K)) return st;
    if (total_M == 0 || I == 0 || G == 0) return FP8BS_OK;
    if (I % 128) return FP8BS_ERR_UNSUPPORTED;  // whole 128-column tiles of h
    if (!offsets_dev || !w3q || !sw3) return FP8BS_ERR_INVALID_ARG;
    if (!h && !hq) return FP8BS_ERR_INVALID_ARG;  // nothing to write
    if (G > kMaxGroups) return FP8BS_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(G) * I > kMaxRows) return FP8BS_ERR_UNSUPPORTED;
    // y's rules apply to h when given; check them with a stand-in otherwise
    if (fp8bs_status st = check_gemm_common(xq, sx, lds, w1q, sw1, total_M, I, K,
                                            h ? h : reinterpret_cast<uint16_t*>(hq), h ? ldh : I))
        return st;
    if (!aligned16(w3q) || (reinterpret_cast<uintptr_t>(sw3) & 3u) || (reinterpret_cast<uintptr_t>(offsets_dev) & 3u))
        return FP8BS_ERR_MISALIGNED;
    if (hq) {
        if (!sh || ldhq < I || ldsh < I / 128) return FP8BS_ERR_INVALID_ARG;
        if (!aligned16(hq) || ldhq % 16 || !aligned16(sh) || ldsh % 4) return FP8BS_ERR_MISALIGNED;
    }
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    GemmArgs a{xq, sx, lds, w1q, sw1, total_M, I, K, h, ldh, offsets_dev, G, nullptr, 0};
    a.wq3 = w3q;
    a.sw3 = sw3;
    a.yq = hq;
    a.ldyq = ldhq;
    a.sy = sh;
    a.ldsy = ldsh;
    return from_cuda(launch_gemm(a, d, cs(stream)));
}

fp8bs_status fp8bs_moe_dispatch(const uint8_t* xq, int64_t ldq, const float* sx, int64_t lds, int64_t tokens,
                                int64_t K, const int32_t* token_of_row, int64_t R, uint8_t* xq_rows,
                                int64_t ldq_rows, float* sx_rows, int64_t lds_rows, fp8bs_stream_t stream) {
    if (tokens < 0 || R < 0) return FP8BS_ERR_INVALID_ARG;
    if (fp8bs_status st = check_k(K)) return st;
    if (R == 0) return FP8BS_OK;
    if (tokens == 0) return FP8BS_ERR_INVALID_ARG;  // no id could be in range
    if (R > kMaxRows || tokens > kMaxRows) return FP8BS_ERR_UNSUPPORTED;
    if (!xq || !sx || !token_of_row || !xq_rows || !sx_rows) return FP8BS_ERR_INVALID_ARG;
    if (ldq < K || ldq_rows < K || lds < K / 128 || lds_rows < K / 128) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(xq) || !aligned16(xq_rows) || ldq % 16 || ldq_rows % 16 ||
        (reinterpret_cast<uintptr_t>(sx) & 3u) || (reinterpret_cast<uintptr_t>(sx_rows) & 3u) ||
        (reinterpret_cast<uintptr_t>(token_of_row) & 3u))
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    return from_cuda(launch_moe_dispatch(xq, ldq, sx, lds, tokens, K, token_of_row, R, xq_rows, ldq_rows, sx_rows,
                                         lds_rows, d, cs(stream)));
}

fp8bs_status fp8bs_moe_combine(const uint16_t* yk, int64_t ldyk, int64_t R, const float* weight_of_row,
                               const int32_t* rows_of_token, int64_t tokens, int32_t topk, int64_t dim,
                               const uint16_t* z, int64_t ldz, uint16_t* y, int64_t ldy, fp8bs_stream_t stream) {
    if (tokens < 0 || topk < 0 || dim < 0 || R < 0) return FP8BS_ERR_INVALID_ARG;
    if (tokens == 0 || dim == 0) return FP8BS_OK;
    if (dim % 8) return FP8BS_ERR_UNSUPPORTED;  // 16-byte chunks of 8 outputs
    if (!y || ldy < dim) return FP8BS_ERR_INVALID_ARG;
    if (topk > 0 && (R == 0 || !yk || !weight_of_row || !rows_of_token || ldyk < dim)) return FP8BS_ERR_INVALID_ARG;
    if (z && ldz < dim) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(y) || ldy % 8) return FP8BS_ERR_MISALIGNED;
    if (topk > 0 && (!aligned16(yk) || ldyk % 8 || (reinterpret_cast<uintptr_t>(weight_of_row) & 3u) ||
                     (reinterpret_cast<uintptr_t>(rows_of_token) & 3u)))
        return FP8BS_ERR_MISALIGNED;
    if (z && (!aligned16(z) || ldz % 8)) return FP8BS_ERR_MISALIGNED;
    if (z && !(z == y && ldz == ldy)) {  // z may be y itself, but no other overlap
        const uintptr_t z0 = reinterpret_cast<uintptr_t>(z), y0 = reinterpret_cast<uintptr_t>(y);
        const uintptr_t z1 = z0 + 2 * static_cast<uintptr_t>((tokens - 1) * ldz + dim);
        const uintptr_t y1 = y0 + 2 * static_cast<uintptr_t>((tokens - 1) * ldy + dim);
        if (z0 < y1 && y0 < z1) return FP8BS_ERR_INVALID_ARG;
    }
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    return from_cuda(launch_moe_combine(yk, ldyk, R, weight_of_row, rows_of_token, tokens, topk, dim, z, ldz, y, ldy,
                                        d, cs(stream)));
}

fp8bs_status fp8bs_moe_gate(const uint16_t* x, int64_t ldx, const uint16_t* wg, const float* bias, int64_t T,
                            int64_t dim, int32_t E, int32_t n_groups, int32_t topk_groups, int32_t top_k,
                            float route_scale, int32_t* ids, float* weights, fp8bs_stream_t stream) {
    if (T < 0 || dim < 0 || E <= 0 || n_groups <= 0 || topk_groups <= 0 || top_k <= 0) return FP8BS_ERR_INVALID_ARG;
    if (E % 16 || E > 256 || dim == 0 || dim % 64) return FP8BS_ERR_UNSUPPORTED;
    if (E % n_groups || n_groups > 32 || topk_groups > n_groups) return FP8BS_ERR_INVALID_ARG;
    if (top_k > 16 || top_k > topk_groups * (E / n_groups)) return FP8BS_ERR_INVALID_ARG;
    if (T == 0) return FP8BS_OK;
    if (T > kMaxRows) return FP8BS_ERR_UNSUPPORTED;
    if (!x || !wg || !ids || !weights || ldx < dim) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(wg) || ldx % 8 || (reinterpret_cast<uintptr_t>(bias) & 3u) ||
        (reinterpret_cast<uintptr_t>(ids) & 3u) || (reinterpret_cast<uintptr_t>(weights) & 3u))
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    return from_cuda(launch_moe_gate(x, ldx, wg, bias, T, dim, E, n_groups, topk_groups, top_k, route_scale, ids,
                                     weights, d, cs(stream)));
}

fp8bs_status fp8bs_moe_route(const int32_t* ids, const float* weights, int64_t T, int32_t top_k, int32_t E,
                             int32_t* offsets, int32_t* token_of_row, int32_t* rows_of_token, float* weight_of_row,
                             fp8bs_stream_t stream) {
    if (T < 0 || top_k <= 0 || E <= 0) return FP8BS_ERR_INVALID_ARG;
    if (E > 256 || top_k > 16) return FP8BS_ERR_UNSUPPORTED;
    if (!offsets) return FP8BS_ERR_INVALID_ARG;
    if (T > 0 && (!ids || !weights || !token_of_row || !rows_of_token || !weight_of_row)) return FP8BS_ERR_INVALID_ARG;
    if (T * static_cast<int64_t>(top_k) > kMaxRows) return FP8BS_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(ids) | reinterpret_cast<uintptr_t>(weights) | reinterpret_cast<uintptr_t>(offsets) |
         reinterpret_cast<uintptr_t>(token_of_row) | reinterpret_cast<uintptr_t>(rows_of_token) |
         reinterpret_cast<uintptr_t>(weight_of_row)) & 3u)
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    return from_cuda(launch_moe_route(ids, weights, T, top_k, E, offsets, token_of_row, rows_of_token, weight_of_row,
                                      d, cs(stream)));
}

fp8bs_status fp8bs_act_quant_cols(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xqt, int64_t ldt,
                                  float* sc, int64_t ldsc, fp8bs_stream_t stream) {
    if (M < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
    if (K % 64) return FP8BS_ERR_UNSUPPORTED;
    if (M == 0 || K == 0) return FP8BS_OK;
    if (M > kMaxRows || K > kMaxRows) return FP8BS_ERR_UNSUPPORTED;
    if (!x || !xqt || !sc) return FP8BS_ERR_INVALID_ARG;
    if (ldx < K || ldt < M || ldsc < K) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xqt) || ldx % 8 || ldt % 16 || (reinterpret_cast<uintptr_t>(sc) & 3u))
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    return from_cuda(launch_act_quant_cols(x, M, K, ldx, xqt, ldt, sc, ldsc, d, cs(stream)));
}

fp8bs_status fp8bs_gemm_wgrad(const uint8_t* dyqt, int64_t lddyt, const float* sdy, int64_t ldsdy, const uint8_t* xqt,
                              int64_t ldxt, const float* sx, int64_t ldsx, int64_t T, int64_t N, int64_t K, float* dw,
                              int64_t lddw, fp8bs_stream_t stream) {
    if (T < 0 || N < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return FP8BS_OK;
    if (T == 0) return FP8BS_ERR_INVALID_ARG;  // an empty sum: no tokens to contract over
    if (T > kMaxRows || N > kMaxRows || K > kMaxRows) return FP8BS_ERR_UNSUPPORTED;
    if (!dyqt || !sdy || !xqt || !sx || !dw) return FP8BS_ERR_INVALID_ARG;
    if (lddyt < T || ldxt < T || ldsdy < N || ldsx < K || lddw < K) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(dyqt) || !aligned16(xqt) || !aligned16(sdy) || !aligned16(sx) || !aligned16(dw) || lddyt % 16 ||
        ldxt % 16 || ldsdy % 4 || ldsx % 4 || lddw % 4)
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    WgradArgs a{dyqt, lddyt, sdy, ldsdy, xqt, ldxt, sx, ldsx, T, N, K, dw, lddw};
    return from_cuda(launch_wgrad(a, d, cs(stream)));
}

fp8bs_status fp8bs_sync_status(fp8bs_stream_t stream) {
    if (cudaStreamSynchronize(cs(stream)) != cudaSuccess) return FP8BS_ERR_CUDA;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    unsigned word = 0;
    if (cudaMemcpyAsync(&word, d.err, sizeof(word), cudaMemcpyDeviceToHost, cs(stream)) != cudaSuccess)
        return FP8BS_ERR_CUDA;
    if (cudaStreamSynchronize(cs(stream)) != cudaSuccess) return FP8BS_ERR_CUDA;
    if (word == 0) return FP8BS_OK;
    if (cudaMemsetAsync(d.err, 0, sizeof(unsigned), cs(stream)) != cudaSuccess) return FP8BS_ERR_CUDA;
    if (cudaStreamSynchronize(cs(stream)) != cudaSuccess) return FP8BS_ERR_CUDA;
    return (word & kDevErrIndex) && !(word & ~kDevErrIndex) ? FP8BS_ERR_INDEX : FP8BS_ERR_TIMEOUT;
}

const char* fp8bs_status_string(fp8bs_status status) {
    switch (status) {
        case FP8BS_OK: return "FP8BS_OK";
        case FP8BS_ERR_INVALID_ARG: return "FP8BS_ERR_INVALID_ARG: null pointer or inconsistent size";
        case FP8BS_ERR_UNSUPPORTED: return "FP8BS_ERR_UNSUPPORTED: K % 128 != 0 or size out of range";
        case FP8BS_ERR_MISALIGNED: return "FP8BS_ERR_MISALIGNED: pointer or leading dimension not 16-byte aligned";
        case FP8BS_ERR_CUDA: return "FP8BS_ERR_CUDA: CUDA runtime error";
        case FP8BS_ERR_TIMEOUT: return "FP8BS_ERR_TIMEOUT: a kernel's bounded wait expired";
        case FP8BS_ERR_INDEX: return "FP8BS_ERR_INDEX: a routed row or token id was out of range";
    }
    return "FP8BS: unknown status";
}

fp8bs_status fp8bs_e4m3_encode_f32(const float* v, int64_t n, uint8_t* q, fp8bs_stream_t stream) {
    if (n < 0) return FP8BS_ERR_INVALID_ARG;
    if (n == 0) return FP8BS_OK;
    if (!v || !q) return FP8BS_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(v) & 3u) return FP8BS_ERR_MISALIGNED;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    return from_cuda(launch_e4m3_encode(v, n, q, d, cs(stream)));
}

fp8bs_status fp8bs_debug_wait_timeout(uint64_t timeout_ns, fp8bs_stream_t stream) {
    if (timeout_ns == 0 || timeout_ns > 10000000000ull) return FP8BS_ERR_INVALID_ARG;
    DeviceInfo d;
    if (fp8bs_status st = device(&d)) return st;
    return from_cuda(launch_wait_selftest(timeout_ns, d, cs(stream)));
}

int fp8bs_version(void) { return (0 << 16) | (1 << 8) | 0; }

}  // extern "C"
