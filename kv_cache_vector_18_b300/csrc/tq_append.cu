// Decode-step append: the step's new key and value rows, one per (batch, KV
// head), quantized straight into the next free token of their cache slabs
// («Шаг 0»–«Шаг 2», and the residual + QJL sketch of «Собственно TurboQuant» for
// a prod handle).  The last block of the launch to finish (a counter in the key
// handle, reset by that block) bumps the lengths — every block has read them by
// then — and zeroes the merge tickets of the decode that follows.
//
// A step appends only B·Hkv rows per side, so the work is latency-bound, not
// bandwidth-bound: one block per (row, side) with four threads per coordinate,
// or, behind a decode with long chunks whose grid leaves SMs free, that many
// blocks looping over the pairs (up to four each).
// Coordinate j forms y_j = Σ_i Π_ji x_i reading Πᵀ down a column (consecutive j
// across a warp, so every load is coalesced), each of its four threads a quarter
// of the sum with all of its loads in flight; the sketch s_i = Σ_j T_ij e_j reads
// T the same way.  K and V share one launch (blockIdx.y picks the side).
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

// Four threads per coordinate: thread (j, q) handles a quarter of every
// contraction, so each thread keeps its D/4 matrix loads in flight at once (one
// round trip to L2 per contraction instead of four).
template <int D>
constexpr int kAppendThreads = 4 * D;

template <int D>
__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // red may still be read from a previous call
    if (lane == 0) red[w] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kAppendThreads<D> / 32; ++k) s += red[k];
    return s;
}

// Σ_k M[k·D + j]·v[k] for coordinate j = threadIdx.x < D: thread (j, q) sums
// k ∈ [qD/4, (q + 1)D/4) with all its loads in flight; the quarters are added in
// order through `part`.  Every thread of the block calls it.
template <int D>
__device__ __forceinline__ float column_dot(const float* __restrict__ M, const float* v, float* part) {
    const int j = threadIdx.x % D, q = threadIdx.x / D;
    constexpr int K = D / 4;
    float p[K];
#pragma unroll
    for (int u = 0; u < K; ++u) p[u] = __ldg(M + (size_t)(q * K + u) * D + j);
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < K; ++u) acc = fmaf(p[u], v[q * K + u], acc);
    part[threadIdx.x] = acc;
    __syncthreads();
    const float r = (part[j] + part[D + j]) + (part[2 * D + j] + part[3 * D + j]);
    __syncthreads();  // part may be reused by the next call
    return r;
}

template <int D, typename TIn>
__device__ __forceinline__ void append_row(const AppendSide& s, int64_t r, int64_t drow, float* xs, float* es,
                                           float* red, float* part, uint32_t* words) {
    const int j = threadIdx.x, lane = j & 31;
    const bool own = j < D;  // threads j < D own coordinate j
    const float xj = own ? load_elem(static_cast<const TIn*>(s.x) + r * D + j) : 0.f;
    if (own) xs[j] = xj;
    const float n = sqrtf(block_sum<D>(xj * xj, red));  // its barriers also publish xs
    const float y = column_dot<D>(s.PiT, xs, part);
    const int idx = own ? bucket_count(s.cb, n, y) : 0;
    if (own && s.b_m > 0) {
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
        const float e = (own && n > 0.f) ? fmaf(y, inv, -s.cb.c[idx]) : 0.f;
        if (own) es[j] = e;
        const float rn = sqrtf(block_sum<D>(e * e, red));
        const float sk = column_dot<D>(s.TT, es, part);
        if (own) {
            const uint32_t bits = __ballot_sync(0xffffffffu, sk >= 0.f);
            if (lane == 0) reinterpret_cast<uint32_t*>(s.out.signs + drow * (int64_t)(D / 8))[j >> 5] = bits;
        }
        if (j == 0) s.out.rnorm[drow] = rn;
    }
}

// LOOP = false: one block per (row, side) pair, grid (rows, 2).  LOOP = true: a
// 1-D grid whose blocks take pairs p = blockIdx.x, blockIdx.x + gridDim.x, …
// (keys for p < rows, values after).
template <int D, typename TIn, bool LOOP>
__global__ void __launch_bounds__(kAppendThreads<D>)
append_rows_kernel(AppendSide k_side, AppendSide v_side, int32_t* __restrict__ lens, int B, int Hkv, int T_max,
                   int rows, int* __restrict__ status, int* __restrict__ done, int* __restrict__ tickets,
                   int n_tickets) {
    __shared__ AppendSide s;
    __shared__ float xs[D];
    __shared__ float es[D];
    __shared__ float red[kAppendThreads<D> / 32];
    __shared__ float part[kAppendThreads<D>];
    __shared__ uint32_t words[D / 8];  // up to 4 bits per coordinate
    __shared__ int s_last;
    // the decode launched after this kernel as its programmatic dependent may start
    // its prologue now; it reads what this kernel writes only after
    // griddepcontrol.wait, i.e. after this grid has completed
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int j = threadIdx.x;
    if constexpr (LOOP) {
        for (int64_t p = blockIdx.x; p < 2 * (int64_t)rows; p += gridDim.x) {
            const bool vside = p >= rows;
            const int64_t r = vside ? p - rows : p;
            __syncthreads();  // the previous pair is done with the shared buffers
            if (j == 0) s = vside ? v_side : k_side;
            if (j < D / 8) words[j] = 0u;
            const int L = lens[r / Hkv];
            if (L >= 0 && L < T_max) {  // block-uniform
                __syncthreads();
                append_row<D, TIn>(s, r, r * T_max + L, xs, es, red, part, words);
            } else if (j == 0 && !vside) {
                atomicExch(status, TQ_STATUS_APPEND_FULL);  // a full slab: the row is not written
            }
        }
    } else {
        const int64_t r = blockIdx.x;
        if (j == 0) s = blockIdx.y == 0 ? k_side : v_side;
        if (j < D / 8) words[j] = 0u;
        const int L = lens[r / Hkv];
        if (L >= 0 && L < T_max) {  // block-uniform
            __syncthreads();
            append_row<D, TIn>(s, r, r * T_max + L, xs, es, red, part, words);
        } else if (j == 0 && blockIdx.y == 0) {
            atomicExch(status, TQ_STATUS_APPEND_FULL);  // a full slab: the row is not written
        }
    }
    // the last block to finish (all blocks have read their lengths by then)
    // bumps every slab that had room and prepares the decode's tickets
    __syncthreads();
    if (j == 0) {
        __threadfence();
        s_last = atomicAdd(done, 1) == (int)(gridDim.x * gridDim.y) - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int b = j; b < B; b += kAppendThreads<D>) {
        const int Lb = lens[b];
        if (Lb >= 0 && Lb < T_max) lens[b] = Lb + 1;
    }
    for (int i = j; i < n_tickets; i += kAppendThreads<D>) tickets[i] = 0;
    if (j == 0) *done = 0;
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
int launch_append_d(const AppendSide& k, const AppendSide& v, int x_dtype, int rows, int B, int Hkv, int T_max,
                    int32_t* lens, int* status, int* done, int* tickets, int n_tickets, int blocks, cudaStream_t st) {
    constexpr int NT = kAppendThreads<D>;
    if (blocks < 2 * rows) {
        if (x_dtype == TQ_BF16)
            append_rows_kernel<D, __nv_bfloat16, true><<<blocks, NT, 0, st>>>(k, v, lens, B, Hkv, T_max, rows, status,
                                                                              done, tickets, n_tickets);
        else
            append_rows_kernel<D, float, true><<<blocks, NT, 0, st>>>(k, v, lens, B, Hkv, T_max, rows, status, done,
                                                                      tickets, n_tickets);
    } else {
        const dim3 grid((unsigned)rows, 2);
        if (x_dtype == TQ_BF16)
            append_rows_kernel<D, __nv_bfloat16, false><<<grid, NT, 0, st>>>(k, v, lens, B, Hkv, T_max, rows, status,
                                                                             done, tickets, n_tickets);
        else
            append_rows_kernel<D, float, false><<<grid, NT, 0, st>>>(k, v, lens, B, Hkv, T_max, rows, status, done,
                                                                     tickets, n_tickets);
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "append launch");
}

}  // namespace

int launch_append(const tq_ctx& hk, const tq_ctx& hv, const void* k_new, const void* v_new, int x_dtype, int B,
                  int Hkv, int T_max, int32_t* lens, const tq_planes& kc, const tq_planes& vc, int* tickets,
                  int n_tickets, int64_t decode_ctas, int decode_chunk, cudaStream_t s) {
    const int64_t rows = (int64_t)B * Hkv;
    if (rows > 0x3fffffffLL) return fail(TQ_EINVAL, "B·Hkv too large");
    // One block per (row, side) pair.  But when the decode's CTAs have long
    // chunks (tens of microseconds of rows below the old length to stream before
    // they need the append) and the SMs the decode grid leaves free can take the
    // pairs at up to four per block, the append runs on those SMs alone and
    // delays no decode CTA.
    const int64_t pairs = 2 * rows, spare = (int64_t)hk.num_sms - decode_ctas;
    const int64_t want = (pairs + 3) / 4;
    const int blocks =
        (int)(decode_chunk >= kAppendStreamChunk && spare >= want && spare < pairs ? spare : pairs);
    const AppendSide k = side_of(hk, k_new, kc), v = side_of(hv, v_new, vc);
    int* done = hk.dp.append_done;
#define TQ_APPEND(DD) \
    return launch_append_d<DD>(k, v, x_dtype, (int)rows, B, Hkv, T_max, lens, hk.dp.status, done, tickets, n_tickets, \
                               blocks, s)
    switch (hk.hp.d) {
        case 32: TQ_APPEND(32);
        case 64: TQ_APPEND(64);
        case 96: TQ_APPEND(96);
        case 128: TQ_APPEND(128);
        case 160: TQ_APPEND(160);
        case 192: TQ_APPEND(192);
        case 224: TQ_APPEND(224);
        case 256: TQ_APPEND(256);
        default: return fail(TQ_EUNSUPPORTED, "d=%d", hk.hp.d);
    }
#undef TQ_APPEND
}

}  // namespace tq
