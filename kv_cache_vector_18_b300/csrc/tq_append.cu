// Decode-step append: the step's new key and value rows, one per (batch, KV
// head), quantized straight into the next free token of their cache slabs
// («Шаг 0»–«Шаг 2», and the residual + QJL sketch of «Собственно TurboQuant» for
// a prod handle), then the lengths bumped.
//
// A step appends only B·Hkv rows per side, so the work is latency-bound, not
// bandwidth-bound: one block per (row, side) with one thread per coordinate.
// Thread j forms y_j = Σ_i Π_ji x_i reading Πᵀ down a column (consecutive j
// across the warp, so every load is coalesced), 32 independent loads in flight
// per batch; the sketch s_i = Σ_j T_ij e_j reads T the same way.  K and V share
// one launch (blockIdx.y picks the side).  Summation orders match the row kernel
// of tq_quantize.cu.
#include "tq_common.cuh"

namespace tq {
namespace {

struct AppendSide {
    const float* PiT;  // [i][j] = Π_ji
    const float* TT;   // [j][i] = (S·Πᵀ)_ij, prod only
    Codebook cb;
    int b_m;
    int prod;
    const void* x;     // [B·Hkv][D] new rows, contiguous
    tq_planes out;
};

template <int D>
__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // red may still be read from a previous call
    if (lane == 0) red[w] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) s += red[k];
    return s;
}

// Σ_k M[k·D + j]·v[k] over k = 0..D−1 in order, 32 loads in flight.
template <int D>
__device__ __forceinline__ float column_dot(const float* __restrict__ M, const float* v, int j) {
    float acc = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < D; k0 += 32) {
        float p[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) p[u] = __ldg(M + (size_t)(k0 + u) * D + j);
#pragma unroll
        for (int u = 0; u < 32; ++u) acc = fmaf(p[u], v[k0 + u], acc);
    }
    return acc;
}

template <int D, typename TIn>
__global__ void __launch_bounds__(D)
append_rows_kernel(AppendSide k_side, AppendSide v_side, const int32_t* __restrict__ lens, int Hkv, int T_max,
                   int* __restrict__ status) {
    __shared__ AppendSide s;
    __shared__ float xs[D];
    __shared__ float es[D];
    __shared__ float red[D / 32];
    __shared__ uint32_t words[D / 8];  // up to 4 bits per coordinate
    const int j = threadIdx.x, lane = j & 31;
    const int64_t r = blockIdx.x;
    if (j == 0) s = blockIdx.y == 0 ? k_side : v_side;
    if (j < D / 8) words[j] = 0u;
    const int L = lens[r / Hkv];
    if (L < 0 || L >= T_max) {  // block-uniform: nothing below runs
        if (j == 0 && blockIdx.y == 0) atomicExch(status, TQ_STATUS_APPEND_FULL);
        return;
    }
    const int64_t drow = r * T_max + L;
    __syncthreads();
    const float xj = load_elem(static_cast<const TIn*>(s.x) + r * D + j);
    xs[j] = xj;
    const float n = sqrtf(block_sum<D>(xj * xj, red));  // its barriers also publish xs
    const float y = column_dot<D>(s.PiT, xs, j);
    const int idx = bucket_count(s.cb, n, y);
    if (s.b_m > 0) {
        const int bit = j * s.b_m, wi = bit >> 5, sh = bit & 31;
        atomicOr(&words[wi], (uint32_t)idx << sh);
        if (sh + s.b_m > 32) atomicOr(&words[wi + 1], (uint32_t)idx >> (32 - sh));
    }
    __syncthreads();
    if (s.b_m > 0 && j < s.b_m * D / 32)
        reinterpret_cast<uint32_t*>(s.out.codes + drow * (int64_t)(s.b_m * D / 8))[j] = words[j];
    if (j == 0) s.out.norm[drow] = n;
    if (s.prod) {
        // e = y/n − c[idx] in the rotated frame; ‖r‖ = ‖e‖ (Π orthogonal); s = T·e
        const float inv = n > 0.f ? 1.f / n : 0.f;
        const float e = n > 0.f ? fmaf(y, inv, -s.cb.c[idx]) : 0.f;
        es[j] = e;
        const float rn = sqrtf(block_sum<D>(e * e, red));
        const float sk = column_dot<D>(s.TT, es, j);
        const uint32_t bits = __ballot_sync(0xffffffffu, sk >= 0.f);
        if (lane == 0) reinterpret_cast<uint32_t*>(s.out.signs + drow * (int64_t)(D / 8))[j >> 5] = bits;
        if (j == 0) s.out.rnorm[drow] = rn;
    }
}

// seq_lens[b] += 1 for every slab that had room (after both sides have read it).
__global__ void bump_lengths_kernel(int32_t* lens, int B, int T_max) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) {
        const int L = lens[b];
        if (L >= 0 && L < T_max) lens[b] = L + 1;
    }
}

AppendSide side_of(const tq_ctx& h, const void* x, const tq_planes& out) {
    AppendSide a;
    a.PiT = h.dp.PiT;
    a.TT = h.dp.TT;
    a.cb = h.cb;
    a.b_m = h.hp.b_mse;
    a.prod = h.hp.variant == TQ_PROD;
    a.x = x;
    a.out = out;
    return a;
}

template <int D>
int launch_append_d(const AppendSide& k, const AppendSide& v, int x_dtype, int rows, int Hkv, int T_max,
                    const int32_t* lens, int* status, cudaStream_t st) {
    const dim3 grid((unsigned)rows, 2);
    if (x_dtype == TQ_BF16)
        append_rows_kernel<D, __nv_bfloat16><<<grid, D, 0, st>>>(k, v, lens, Hkv, T_max, status);
    else
        append_rows_kernel<D, float><<<grid, D, 0, st>>>(k, v, lens, Hkv, T_max, status);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "append launch");
}

}  // namespace

int launch_append(const tq_ctx& hk, const tq_ctx& hv, const void* k_new, const void* v_new, int x_dtype, int B,
                  int Hkv, int T_max, int32_t* lens, const tq_planes& kc, const tq_planes& vc, cudaStream_t s) {
    const int64_t rows = (int64_t)B * Hkv;
    if (rows > 0x7fffffffLL) return fail(TQ_EINVAL, "B·Hkv too large");
    const AppendSide k = side_of(hk, k_new, kc), v = side_of(hv, v_new, vc);
    int rc;
    switch (hk.hp.d) {
        case 32: rc = launch_append_d<32>(k, v, x_dtype, (int)rows, Hkv, T_max, lens, hk.dp.status, s); break;
        case 64: rc = launch_append_d<64>(k, v, x_dtype, (int)rows, Hkv, T_max, lens, hk.dp.status, s); break;
        case 96: rc = launch_append_d<96>(k, v, x_dtype, (int)rows, Hkv, T_max, lens, hk.dp.status, s); break;
        case 128: rc = launch_append_d<128>(k, v, x_dtype, (int)rows, Hkv, T_max, lens, hk.dp.status, s); break;
        case 160: rc = launch_append_d<160>(k, v, x_dtype, (int)rows, Hkv, T_max, lens, hk.dp.status, s); break;
        case 192: rc = launch_append_d<192>(k, v, x_dtype, (int)rows, Hkv, T_max, lens, hk.dp.status, s); break;
        case 224: rc = launch_append_d<224>(k, v, x_dtype, (int)rows, Hkv, T_max, lens, hk.dp.status, s); break;
        case 256: rc = launch_append_d<256>(k, v, x_dtype, (int)rows, Hkv, T_max, lens, hk.dp.status, s); break;
        default: return fail(TQ_EUNSUPPORTED, "d=%d", hk.hp.d);
    }
    if (rc != TQ_OK) return rc;
    bump_lengths_kernel<<<(B + 127) / 128, 128, 0, s>>>(lens, B, T_max);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "sequence length update");
}

}  // namespace tq
