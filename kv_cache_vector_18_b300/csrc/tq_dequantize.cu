// tq_dequantize: Q⁻¹ of «Шаг 2» (centroids rotated back by Πᵀ) plus, for prod,
// the QJL reconstruction √(π/2)/d·‖r‖·Sᵀz of «QJL» / «Собственно TurboQuant».
// One warp per row; lane l produces output coordinates i = l + 32m.
#include "tq_common.cuh"

namespace tq {
namespace {

constexpr int kWarps = 8;

template <int D, bool PROD, typename TOut>
__global__ void __launch_bounds__(kWarps * 32)
dequantize_rows_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ signs,
                       const float* __restrict__ norm, const float* __restrict__ rnorm, int64_t n_rows,
                       const float* __restrict__ Pi, const float* __restrict__ S, Codebook cb, int b_m,
                       float gamma, TOut* __restrict__ y, ChannelMap cm) {
    constexpr int PER = D / 32;
    __shared__ float cs[kWarps][D];
    __shared__ float zs[kWarps][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
    if (row >= n_rows) return;

    const uint32_t* cw = reinterpret_cast<const uint32_t*>(codes + row * (int64_t)(b_m * D / 8));
#pragma unroll
    for (int m = 0; m < PER; ++m) {
        const int j = lane + 32 * m;
        cs[warp][j] = b_m > 0 ? cb.c[read_code(cw, j, b_m)] : 0.f;
        if constexpr (PROD) {
            const uint32_t sw = reinterpret_cast<const uint32_t*>(signs + row * (int64_t)(D / 8))[m];
            zs[warp][j] = ((sw >> lane) & 1u) ? 1.f : -1.f;
        }
    }
    __syncwarp();
    const float n = norm[row];
    const float qs = PROD ? gamma * rnorm[row] : 0.f;
    const int64_t ystride = cm.ch != nullptr ? cm.d_full : D;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
        const int i = lane + 32 * m;
        float a = 0.f, b = 0.f;
        for (int j = 0; j < D; ++j) {
            a = fmaf(__ldg(Pi + (size_t)j * D + i), cs[warp][j], a);
            if constexpr (PROD) b = fmaf(__ldg(S + (size_t)j * D + i), zs[warp][j], b);
        }
        const float v = n * fmaf(qs, b, a);
        const int64_t o = row * ystride + channel_of(cm, i);
        if constexpr (sizeof(TOut) == 4)
            y[o] = v;
        else
            y[o] = __float2bfloat16_rn(v);
    }
}

template <int D>
int launch_d(const tq_ctx& h, const tq_planes& in, int64_t n_rows, void* y, int y_dtype, cudaStream_t s,
             ChannelMap cm = ChannelMap()) {
    const int64_t blocks = (n_rows + kWarps - 1) / kWarps;
    if (blocks > 0x7fffffffLL) return fail(TQ_EINVAL, "n_rows too large");
    dim3 grid((unsigned)blocks), block(kWarps * 32);
    const bool prod = h.hp.variant == TQ_PROD;
#define TQ_DQ(P, T) \
    dequantize_rows_kernel<D, P, T><<<grid, block, 0, s>>>(in.codes, in.signs, in.norm, in.rnorm, n_rows, h.dp.Pi, \
                                                           h.dp.S, h.cb, h.hp.b_mse, h.gamma, static_cast<T*>(y), cm)
    if (y_dtype == TQ_F32) {
        if (prod) TQ_DQ(true, float); else TQ_DQ(false, float);
    } else {
        if (prod) TQ_DQ(true, __nv_bfloat16); else TQ_DQ(false, __nv_bfloat16);
    }
#undef TQ_DQ
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "dequantize launch");
}

}  // namespace

int launch_dequantize_part(const tq_ctx& h, const tq_planes& in, int64_t n_rows, const int32_t* ch, int d_full,
                           void* y, int y_dtype, cudaStream_t s) {
    ChannelMap cm;
    cm.ch = ch;
    cm.d_full = d_full;
    cm.status = h.dp.status;
    switch (h.hp.d) {
        case 32: return launch_d<32>(h, in, n_rows, y, y_dtype, s, cm);
        case 64: return launch_d<64>(h, in, n_rows, y, y_dtype, s, cm);
        case 96: return launch_d<96>(h, in, n_rows, y, y_dtype, s, cm);
        case 128: return launch_d<128>(h, in, n_rows, y, y_dtype, s, cm);
        case 160: return launch_d<160>(h, in, n_rows, y, y_dtype, s, cm);
        case 192: return launch_d<192>(h, in, n_rows, y, y_dtype, s, cm);
        case 224: return launch_d<224>(h, in, n_rows, y, y_dtype, s, cm);
        default: return fail(TQ_EUNSUPPORTED, "part d=%d", h.hp.d);
    }
}

int launch_dequantize(const tq_ctx& h, const tq_planes& in, int64_t n_rows, void* y, int y_dtype, cudaStream_t s) {
    switch (h.hp.d) {
        case 32: return launch_d<32>(h, in, n_rows, y, y_dtype, s);
        case 64: return launch_d<64>(h, in, n_rows, y, y_dtype, s);
        case 96: return launch_d<96>(h, in, n_rows, y, y_dtype, s);
        case 128: return launch_d<128>(h, in, n_rows, y, y_dtype, s);
        case 160: return launch_d<160>(h, in, n_rows, y, y_dtype, s);
        case 192: return launch_d<192>(h, in, n_rows, y, y_dtype, s);
        case 224: return launch_d<224>(h, in, n_rows, y, y_dtype, s);
        case 256: return launch_d<256>(h, in, n_rows, y, y_dtype, s);
        default: return fail(TQ_EUNSUPPORTED, "d=%d", h.hp.d);
    }
}

}  // namespace tq
