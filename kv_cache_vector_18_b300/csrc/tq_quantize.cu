// tq_quantize: TurboQuant row quantization («Шаг 0»–«Шаг 2», and the prod
// residual + QJL sketch of «Собственно TurboQuant»).
//
// Straightforward CUDA-core formulation: one warp per row, lane l owns rotated
// coordinates j = l + 32m.  y = Π·x in fp32 FMA against ΠᵀΠ-layout rows cached
// in L1/L2; bucketize against norm-scaled boundaries; pack through shared words.
#include "tq_common.cuh"

namespace tq {
namespace {

constexpr int kWarps = 8;

template <int D, bool PROD, typename TIn>
__global__ void __launch_bounds__(kWarps * 32)
quantize_rows_kernel(const TIn* __restrict__ x, int64_t n_rows, int64_t stride,
                     const float* __restrict__ PiT, const float* __restrict__ TT, Codebook cb,
                     int b_m, uint8_t* __restrict__ codes, uint8_t* __restrict__ signs,
                     float* __restrict__ norm_out, float* __restrict__ rnorm_out, ChannelMap cm) {
    constexpr int PER = D / 32;
    __shared__ float xs[kWarps][D];
    __shared__ uint32_t words[kWarps][D * 4 / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
    if (row >= n_rows) return;  // whole warp exits together; no block barriers below

    const TIn* xr = x + row * stride;
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
        float v = load_elem(xr + channel_of(cm, lane + 32 * m));
        xs[warp][lane + 32 * m] = v;
        ss = fmaf(v, v, ss);
    }
    const float n = sqrtf(warp_sum(ss));
    for (int w = lane; w < D * 4 / 32; w += 32) words[warp][w] = 0u;
    __syncwarp();

    float y[PER];
#pragma unroll
    for (int m = 0; m < PER; ++m) y[m] = 0.f;
    for (int i = 0; i < D; ++i) {
        const float xi = xs[warp][i];
#pragma unroll
        for (int m = 0; m < PER; ++m) y[m] = fmaf(__ldg(PiT + (size_t)i * D + lane + 32 * m), xi, y[m]);
    }

    int idx[PER];
#pragma unroll
    for (int m = 0; m < PER; ++m) idx[m] = bucket_count(cb, n, y[m]);

    if (b_m > 0) {
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            const int bit = (lane + 32 * m) * b_m;
            const int wi = bit >> 5, sh = bit & 31;
            atomicOr(&words[warp][wi], (uint32_t)idx[m] << sh);
            if (sh + b_m > 32) atomicOr(&words[warp][wi + 1], (uint32_t)idx[m] >> (32 - sh));
        }
        __syncwarp();
        const int nw = b_m * D / 32;
        uint32_t* dst = reinterpret_cast<uint32_t*>(codes + row * (int64_t)(b_m * D / 8));
        for (int w = lane; w < nw; w += 32) dst[w] = words[warp][w];
    }
    if (lane == 0) norm_out[row] = n;

    if constexpr (PROD) {
        // Residual in the rotated frame, e = y/n − c[idx]; ‖r‖ = ‖e‖ since Π is orthogonal.
        const float inv = n > 0.f ? 1.f / n : 0.f;
        float e[PER], es = 0.f;
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            e[m] = n > 0.f ? fmaf(y[m], inv, -cb.c[idx[m]]) : 0.f;
            es = fmaf(e[m], e[m], es);
        }
        __syncwarp();
#pragma unroll
        for (int m = 0; m < PER; ++m) xs[warp][lane + 32 * m] = e[m];
        __syncwarp();
        const float rn = sqrtf(warp_sum(es));
        // S·r = S·Πᵀ·e = T·e; sign bit i = [(T e)_i ≥ 0]
        float s[PER];
#pragma unroll
        for (int m = 0; m < PER; ++m) s[m] = 0.f;
        for (int j = 0; j < D; ++j) {
            const float ej = xs[warp][j];
#pragma unroll
            for (int m = 0; m < PER; ++m) s[m] = fmaf(__ldg(TT + (size_t)j * D + lane + 32 * m), ej, s[m]);
        }
        uint32_t* sdst = reinterpret_cast<uint32_t*>(signs + row * (int64_t)(D / 8));
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            const uint32_t bits = __ballot_sync(0xffffffffu, s[m] >= 0.f);
            if (lane == 0) sdst[m] = bits;
        }
        if (lane == 0) rnorm_out[row] = rn;
    }
}

template <int D>
int launch_d(const tq_ctx& h, const void* x, int x_dtype, int64_t n_rows, int64_t stride,
             const tq_planes& out, cudaStream_t s, ChannelMap cm = ChannelMap()) {
    const int64_t blocks = (n_rows + kWarps - 1) / kWarps;
    if (blocks > 0x7fffffffLL) return fail(TQ_EINVAL, "n_rows too large");
    dim3 grid((unsigned)blocks), block(kWarps * 32);
    const bool prod = h.hp.variant == TQ_PROD;
    if (x_dtype == TQ_BF16) {
        auto xp = static_cast<const __nv_bfloat16*>(x);
        if (prod)
            quantize_rows_kernel<D, true><<<grid, block, 0, s>>>(xp, n_rows, stride, h.dp.PiT, h.dp.TT, h.cb, h.hp.b_mse,
                                                                 out.codes, out.signs, out.norm, out.rnorm, cm);
        else
            quantize_rows_kernel<D, false><<<grid, block, 0, s>>>(xp, n_rows, stride, h.dp.PiT, h.dp.TT, h.cb, h.hp.b_mse,
                                                                  out.codes, out.signs, out.norm, out.rnorm, cm);
    } else {
        auto xp = static_cast<const float*>(x);
        if (prod)
            quantize_rows_kernel<D, true><<<grid, block, 0, s>>>(xp, n_rows, stride, h.dp.PiT, h.dp.TT, h.cb, h.hp.b_mse,
                                                                 out.codes, out.signs, out.norm, out.rnorm, cm);
        else
            quantize_rows_kernel<D, false><<<grid, block, 0, s>>>(xp, n_rows, stride, h.dp.PiT, h.dp.TT, h.cb, h.hp.b_mse,
                                                                  out.codes, out.signs, out.norm, out.rnorm, cm);
    }
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "quantize launch");
}

}  // namespace

int launch_quantize_part(const tq_ctx& h, const void* x, int x_dtype, int64_t n_rows, int64_t stride,
                         const int32_t* ch, int d_full, const tq_planes& out, cudaStream_t s) {
    ChannelMap cm;
    cm.ch = ch;
    cm.d_full = d_full;
    cm.status = h.dp.status;
    switch (h.hp.d) {
        case 32: return launch_d<32>(h, x, x_dtype, n_rows, stride, out, s, cm);
        case 64: return launch_d<64>(h, x, x_dtype, n_rows, stride, out, s, cm);
        case 96: return launch_d<96>(h, x, x_dtype, n_rows, stride, out, s, cm);
        case 128: return launch_d<128>(h, x, x_dtype, n_rows, stride, out, s, cm);
        case 160: return launch_d<160>(h, x, x_dtype, n_rows, stride, out, s, cm);
        case 192: return launch_d<192>(h, x, x_dtype, n_rows, stride, out, s, cm);
        case 224: return launch_d<224>(h, x, x_dtype, n_rows, stride, out, s, cm);
        default: return fail(TQ_EUNSUPPORTED, "part d=%d", h.hp.d);
    }
}

int launch_quantize(const tq_ctx& h, const void* x, int x_dtype, int64_t n_rows, int64_t stride,
                    const tq_planes& out, cudaStream_t s) {
    if (quantize_tc_supported(h, x_dtype, n_rows)) return launch_quantize_tc(h, x, x_dtype, n_rows, stride, out, s);
    switch (h.hp.d) {
        case 32: return launch_d<32>(h, x, x_dtype, n_rows, stride, out, s);
        case 64: return launch_d<64>(h, x, x_dtype, n_rows, stride, out, s);
        case 96: return launch_d<96>(h, x, x_dtype, n_rows, stride, out, s);
        case 128: return launch_d<128>(h, x, x_dtype, n_rows, stride, out, s);
        case 160: return launch_d<160>(h, x, x_dtype, n_rows, stride, out, s);
        case 192: return launch_d<192>(h, x, x_dtype, n_rows, stride, out, s);
        case 224: return launch_d<224>(h, x, x_dtype, n_rows, stride, out, s);
        case 256: return launch_d<256>(h, x, x_dtype, n_rows, stride, out, s);
        default: return fail(TQ_EUNSUPPORTED, "d=%d", h.hp.d);
    }
}

}  // namespace tq
