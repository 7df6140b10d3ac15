// tq_decode_attention: decode attention read straight from the packed cache.
//
// Math (see include/tq.h): the query is rotated once (q′ = Π_k q, q″ = S_k q),
// each cached key is scored by codebook lookup plus the QJL correction, and
// values are accumulated in their rotated frame (plus, for prod values, in the
// S frame) so that Π_vᵀ (and S_vᵀ) is applied once per output head.
//
// Three launches: query prep, split-K flash-decoding over token chunks with an
// online softmax per split, and a merge that combines the splits and un-rotates.
// For d = 128 the split step runs on the tensor cores (tq_decode_mma.cuh); the
// CUDA-core split kernel below serves every other head dimension.
#include <math.h>

#include "tq_common.cuh"
#include "tq_decode_args.h"

namespace tq {
namespace {

constexpr int kSplitWarps = 4;
constexpr int kMinChunk = 64;
constexpr int64_t kMaxChunk = 8192;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// d = 128 runs the tensor-core split kernel (tq_decode_mma.cuh)
constexpr bool use_mma_split(int d) { return d == mmadec::D128; }

struct WsLayout {
    size_t qr, qs, pm, pl, pacc, pacc2, cnt, total;
};

WsLayout ws_layout(const DecodeShape& p, bool vprod) {
    WsLayout w;
    const size_t heads = (size_t)p.B * p.Hq;
    size_t off = 0;
    w.qr = off;
    off = align256(off + heads * p.d * 4);
    w.qs = off;
    off = align256(off + heads * p.d * 4);
    w.pm = off;
    off = align256(off + heads * p.n_splits * 4);
    w.pl = off;
    off = align256(off + heads * p.n_splits * 4);
    w.pacc = off;
    off = align256(off + heads * p.n_splits * p.d * 4);
    w.pacc2 = off;
    if (vprod) off = align256(off + heads * p.n_splits * p.d * 4);
    w.cnt = off;  // one ticket per (batch, KV head, head block): at most B·Hq
    off = align256(off + heads * 4);
    w.total = off;
    return w;
}

template <int D, bool KPROD, typename TQ>
__global__ void query_prep_kernel(const TQ* __restrict__ q, const float* __restrict__ PiT,
                                  const float* __restrict__ ST, int Hq, float* __restrict__ qr,
                                  float* __restrict__ qs, int* __restrict__ cnt, int ncnt) {
    __shared__ float qv[D];
    const int h = blockIdx.x, b = blockIdx.y, j = threadIdx.x;
    // zero the split-merge tickets of this call
    const int gt = (blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
    if (gt < ncnt) cnt[gt] = 0;
    const size_t base = ((size_t)b * Hq + h) * D;
    qv[j] = load_elem(q + base + j);
    __syncthreads();
    float a = 0.f, c = 0.f;
    for (int i = 0; i < D; ++i) {
        a = fmaf(__ldg(PiT + (size_t)i * D + j), qv[i], a);
        if constexpr (KPROD) c = fmaf(__ldg(ST + (size_t)i * D + j), qv[i], c);
    }
    qr[base + j] = a;
    if constexpr (KPROD) qs[base + j] = c;
}

template <int D, bool KPROD, bool VPROD>
__global__ void __launch_bounds__(kSplitWarps * 32)
decode_split_kernel(const SplitArgs a) {
    constexpr int PER = D / 32;
    extern __shared__ float sm[];
    // This CTA serves query heads [hb·kMaxGroup, hb·kMaxGroup + G) of its KV head's group.
    const int hb = blockIdx.y % a.n_hblocks, kvh = blockIdx.y / a.n_hblocks;
    const int G = min(kMaxGroup, a.G - hb * kMaxGroup);
    float* qr = sm;                                   // [G][D]
    float* qs = qr + G * D;                           // [G][D]
    float* acc = qs + G * D;                          // [warps][G][D]
    float* acc2 = acc + kSplitWarps * G * D;          // [warps][G][D] (prod values)
    float* wm = acc2 + (VPROD ? kSplitWarps * G * D : 0);  // [warps][G]
    float* wl = wm + kSplitWarps * G;                 // [warps][G]

    const int split = blockIdx.x, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int L = a.seq_lens[b];
    L = L < 0 ? 0 : (L > a.T_max ? a.T_max : L);
    const int t0 = split * a.chunk;
    const int t1 = min(t0 + a.chunk, L);
    const size_t head0 = (size_t)b * a.Hq + (size_t)kvh * a.G + (size_t)hb * kMaxGroup;

    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
        qr[i] = a.qr[head0 * D + i];
        if (KPROD) qs[i] = a.qs[head0 * D + i];
    }
    for (int i = threadIdx.x; i < kSplitWarps * G * D; i += blockDim.x) {
        acc[i] = 0.f;
        if (VPROD) acc2[i] = 0.f;
    }
    __syncthreads();

    float m_[kMaxGroup], l_[kMaxGroup];
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
        m_[h] = -INFINITY;
        l_[h] = 0.f;
    }
    float* myacc = acc + warp * G * D;
    float* myacc2 = acc2 + warp * G * D;
    const int kcb = a.kb * D / 8, vcb = a.vb * D / 8;

    for (int t = t0 + warp; t < t1; t += kSplitWarps) {
        const int64_t row = ((int64_t)b * a.Hkv + kvh) * a.T_max + t;
        float ck[PER], zk[PER];
        const uint32_t* kw = reinterpret_cast<const uint32_t*>(a.kcodes + row * kcb);
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            ck[m] = a.kb > 0 ? a.kcb.c[read_code(kw, lane + 32 * m, a.kb)] : 0.f;
            if (KPROD) {
                const uint32_t sw = reinterpret_cast<const uint32_t*>(a.ksigns + row * (D / 8))[m];
                zk[m] = ((sw >> lane) & 1u) ? 1.f : -1.f;
            }
        }
        const float kn = a.knorm[row];
        const float krn = KPROD ? a.kgamma * a.krnorm[row] : 0.f;

        float cv[PER], zv[PER];
        const uint32_t* vw = reinterpret_cast<const uint32_t*>(a.vcodes + row * vcb);
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            cv[m] = a.vb > 0 ? a.vcb.c[read_code(vw, lane + 32 * m, a.vb)] : 0.f;
            if (VPROD) {
                const uint32_t sw = reinterpret_cast<const uint32_t*>(a.vsigns + row * (D / 8))[m];
                zv[m] = ((sw >> lane) & 1u) ? 1.f : -1.f;
            }
        }
        const float vn = a.vnorm[row];
        const float vrn = VPROD ? a.vgamma * a.vrnorm[row] : 0.f;

        for (int h = 0; h < G; ++h) {
            float part = 0.f, partz = 0.f;
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                part = fmaf(qr[h * D + lane + 32 * m], ck[m], part);
                if (KPROD) partz = fmaf(qs[h * D + lane + 32 * m], zk[m], partz);
            }
            part = warp_sum(fmaf(krn, partz, part));
            const float s = a.scale * kn * part;
            if (a.scores != nullptr && lane == 0) a.scores[(head0 + h) * a.T_max + t] = s;
            // online softmax (all lanes hold identical values)
            float mh = m_[0], lh = l_[0];
#pragma unroll
            for (int k = 1; k < kMaxGroup; ++k)
                if (k == h) { mh = m_[k]; lh = l_[k]; }
            const float mn = fmaxf(mh, s);
            const float corr = __expf(mh - mn);
            const float p = __expf(s - mn);
            lh = fmaf(lh, corr, p);
#pragma unroll
            for (int k = 0; k < kMaxGroup; ++k)
                if (k == h) { m_[k] = mn; l_[k] = lh; }
            const float pv = p * vn;
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                float* r = myacc + h * D + lane + 32 * m;
                *r = fmaf(*r, corr, pv * cv[m]);
                if (VPROD) {
                    float* r2 = myacc2 + h * D + lane + 32 * m;
                    *r2 = fmaf(*r2, corr, pv * vrn * zv[m]);
                }
            }
        }
    }
    if (lane == 0)
        for (int h = 0; h < G; ++h) {
            float mh = m_[0], lh = l_[0];
#pragma unroll
            for (int k = 1; k < kMaxGroup; ++k)
                if (k == h) { mh = m_[k]; lh = l_[k]; }
            wm[warp * G + h] = mh;
            wl[warp * G + h] = lh;
        }
    __syncthreads();

    // Combine the warps of this split, write the split's partial state.
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
        const int h = i / D;
        float M = -INFINITY;
        for (int w = 0; w < kSplitWarps; ++w) M = fmaxf(M, wm[w * G + h]);
        float o = 0.f, o2 = 0.f, l = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < kSplitWarps; ++w) {
                const float f = __expf(wm[w * G + h] - M);
                o = fmaf(f, acc[w * G * D + i], o);
                if (VPROD) o2 = fmaf(f, acc2[w * G * D + i], o2);
                l = fmaf(f, wl[w * G + h], l);
            }
        }
        const size_t ps = (head0 + h) * a.n_splits + split;
        a.pacc[ps * D + (i % D)] = o;
        if (VPROD) a.pacc2[ps * D + (i % D)] = o2;
        if (i % D == 0) {
            a.pm[ps] = M;
            a.pl[ps] = l;
        }
    }
}

template <int D, bool VPROD>
__global__ void decode_merge_kernel(const float* __restrict__ pm, const float* __restrict__ pl,
                                    const float* __restrict__ pacc, const float* __restrict__ pacc2,
                                    const float* __restrict__ Pi, const float* __restrict__ S, int Hq,
                                    int n_splits, float* __restrict__ out) {
    __shared__ float o1[D], o2[D];
    const int h = blockIdx.x, b = blockIdx.y, j = threadIdx.x;
    const size_t head = (size_t)b * Hq + h;
    float M = -INFINITY;
    for (int s = 0; s < n_splits; ++s) M = fmaxf(M, pm[head * n_splits + s]);
    float a = 0.f, c = 0.f, l = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < n_splits; ++s) {
            const size_t ps = head * n_splits + s;
            const float f = __expf(pm[ps] - M);
            l = fmaf(f, pl[ps], l);
            a = fmaf(f, pacc[ps * D + j], a);
            if (VPROD) c = fmaf(f, pacc2[ps * D + j], c);
        }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    o1[j] = a * inv;
    o2[j] = c * inv;
    __syncthreads();
    // out = Π_vᵀ o1 (+ S_vᵀ o2): out_i = Σ_j Π_ji o1_j
    float r = 0.f;
    for (int k = 0; k < D; ++k) {
        r = fmaf(__ldg(Pi + (size_t)k * D + j), o1[k], r);
        if (VPROD) r = fmaf(__ldg(S + (size_t)k * D + j), o2[k], r);
    }
    out[head * D + j] = r;
}

// The tensor-core split kernel is written for d = 128 (the head dimension of
// every workload this library is tuned for).

int launch_split_mma_any(const SplitArgs& a, dim3 grid, int kb, bool kp, int vb, bool vp, bool pdl, cudaStream_t s) {
    using namespace mmadec;
    if (kp) {
        switch (kb) {
            case 0: return launch_for_k<0, true>(a, grid, vb, vp, pdl, s);
            case 1: return launch_for_k<1, true>(a, grid, vb, vp, pdl, s);
            case 2: return launch_for_k<2, true>(a, grid, vb, vp, pdl, s);
            case 3: return launch_for_k<3, true>(a, grid, vb, vp, pdl, s);
            default: break;
        }
    } else {
        switch (kb) {
            case 1: return launch_for_k<1, false>(a, grid, vb, vp, pdl, s);
            case 2: return launch_for_k<2, false>(a, grid, vb, vp, pdl, s);
            case 3: return launch_for_k<3, false>(a, grid, vb, vp, pdl, s);
            case 4: return launch_for_k<4, false>(a, grid, vb, vp, pdl, s);
            default: break;
        }
    }
    return fail(TQ_EUNSUPPORTED, "tensor-core decode: key b_m=%d", kb);
}

// Zeroes the split-merge tickets of the decode launched after it, which is its
// programmatic dependent and may start right away; this grid completes only once
// every kernel before it has, so the decode's griddepcontrol.wait covers them
// all.  Launched itself as a programmatic dependent, its zeroing may overlap the
// kernel before it, which therefore must not use this workspace (the quantize
// kernels do not; a decode never lets its dependents start early).
__global__ void clear_tickets_kernel(int* __restrict__ tickets, int n) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) tickets[i] = 0;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

int launch_clear_tickets(int* tickets, int n, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, clear_tickets_kernel, tickets, n);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "clearing the split tickets");
}

namespace {

template <int D>
int launch_d(const tq_ctx& hk, const tq_ctx& hv, const DecodeShape& p, const void* q, int q_dtype,
             const tq_planes& kc, const tq_planes& vc, const int32_t* seq_lens, float scale, float* out,
             float* scores, void* workspace, cudaStream_t s, bool tickets_zeroed) {
    const bool kprod = hk.hp.variant == TQ_PROD, vprod = hv.hp.variant == TQ_PROD;
    const WsLayout w = ws_layout(p, vprod);
    char* ws = static_cast<char*>(workspace);
    float* qr = reinterpret_cast<float*>(ws + w.qr);
    float* qs = reinterpret_cast<float*>(ws + w.qs);
    int* cnt = reinterpret_cast<int*>(ws + w.cnt);
    dim3 pg(p.Hq, p.B);
    cudaError_t e = cudaSuccess;
    SplitArgs a;
    a.kcodes = kc.codes; a.ksigns = kc.signs; a.knorm = kc.norm; a.krnorm = kc.rnorm;
    a.vcodes = vc.codes; a.vsigns = vc.signs; a.vnorm = vc.norm; a.vrnorm = vc.rnorm;
    a.seq_lens = seq_lens; a.qr = qr; a.qs = qs;
    a.pm = reinterpret_cast<float*>(ws + w.pm);
    a.pl = reinterpret_cast<float*>(ws + w.pl);
    a.pacc = reinterpret_cast<float*>(ws + w.pacc);
    a.pacc2 = reinterpret_cast<float*>(ws + w.pacc2);
    a.scores = scores;
    a.kcb = hk.cb; a.vcb = hv.cb; a.kb = hk.hp.b_mse; a.vb = hv.hp.b_mse;
    a.kgamma = hk.gamma; a.vgamma = hv.gamma; a.scale = scale;
    a.B = p.B; a.Hq = p.Hq; a.Hkv = p.Hkv; a.T_max = p.T_max; a.G = p.G;
    a.n_splits = p.n_splits; a.chunk = p.chunk;
    a.cnt = cnt; a.vPi = hv.dp.Pi; a.vS = hv.dp.S; a.out = out;
    a.vPiT_hi = hv.dp.PiT_hi; a.vPiT_lo = hv.dp.PiT_lo; a.vST_hi = hv.dp.ST_hi; a.vST_lo = hv.dp.ST_lo;
    a.q = q; a.q_f32 = q_dtype == TQ_F32; a.kPi_hi = hk.dp.Pi_hi; a.kPi_lo = hk.dp.Pi_lo; a.kS_hi = hk.dp.S_hi; a.kS_lo = hk.dp.S_lo;
    a.status = hk.dp.status;
    if (use_mma_split(D)) {
        // query rotation, split and merge all happen in the split kernel
        a.n_hblocks = (p.G + mmadec::kHeadsPerCta - 1) / mmadec::kHeadsPerCta;
        // the kernel is the programmatic dependent of the decode-step append (which
        // cleared the tickets and does not write q) or of the ticket clearing
        // kernel: its prologue overlaps the kernels before it
        a.after_append = tickets_zeroed ? 1 : 0;
        if (!tickets_zeroed) {
            const int rc = launch_clear_tickets(cnt, p.B * p.Hq, s);
            if (rc != TQ_OK) return rc;
        }
        return launch_split_mma_any(a, dim3(p.B, p.Hkv * a.n_hblocks, p.n_splits), hk.hp.b_mse, kprod, hv.hp.b_mse,
                                    vprod, true, s);
    }

    // CUDA-core path: query prep (which also clears the tickets), split, merge
    if (q_dtype == TQ_F32) {
        auto qp = static_cast<const float*>(q);
        if (kprod) query_prep_kernel<D, true><<<pg, D, 0, s>>>(qp, hk.dp.PiT, hk.dp.ST, p.Hq, qr, qs, cnt, (int)((size_t)p.B * p.Hq));
        else query_prep_kernel<D, false><<<pg, D, 0, s>>>(qp, hk.dp.PiT, hk.dp.ST, p.Hq, qr, qs, cnt, (int)((size_t)p.B * p.Hq));
    } else {
        auto qp = static_cast<const __nv_bfloat16*>(q);
        if (kprod) query_prep_kernel<D, true><<<pg, D, 0, s>>>(qp, hk.dp.PiT, hk.dp.ST, p.Hq, qr, qs, cnt, (int)((size_t)p.B * p.Hq));
        else query_prep_kernel<D, false><<<pg, D, 0, s>>>(qp, hk.dp.PiT, hk.dp.ST, p.Hq, qr, qs, cnt, (int)((size_t)p.B * p.Hq));
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "query prep launch");

    a.n_hblocks = (p.G + kMaxGroup - 1) / kMaxGroup;
    const int gmax = p.G < kMaxGroup ? p.G : kMaxGroup;
    const size_t smem = sizeof(float) * ((size_t)gmax * D * (2 + kSplitWarps * (vprod ? 2 : 1)) + 2 * kSplitWarps * gmax);
    dim3 sg(p.n_splits, p.Hkv * a.n_hblocks, p.B);
#define TQ_SPLIT(KP, VP)                                                                              \
    do {                                                                                              \
        auto fn = decode_split_kernel<D, KP, VP>;                                                     \
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);        \
        if (e != cudaSuccess) return cuda_fail(e, "decode smem attribute");                          \
        fn<<<sg, kSplitWarps * 32, smem, s>>>(a);                                                     \
    } while (0)
    if (kprod && vprod) TQ_SPLIT(true, true);
    else if (kprod) TQ_SPLIT(true, false);
    else if (vprod) TQ_SPLIT(false, true);
    else TQ_SPLIT(false, false);
#undef TQ_SPLIT
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "decode split launch");

    if (vprod)
        decode_merge_kernel<D, true><<<pg, D, 0, s>>>(a.pm, a.pl, a.pacc, a.pacc2, hv.dp.Pi, hv.dp.S, p.Hq,
                                                      p.n_splits, out);
    else
        decode_merge_kernel<D, false><<<pg, D, 0, s>>>(a.pm, a.pl, a.pacc, a.pacc2, hv.dp.Pi, hv.dp.S, p.Hq,
                                                       p.n_splits, out);
    e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "decode merge launch");
}

}  // namespace

int decode_plan(const tq_ctx& hk, const tq_ctx& hv, int B, int Hq, int Hkv, int T_max, DecodeShape* plan,
                size_t* ws_bytes) {
    if (hk.hp.d != hv.hp.d) return fail(TQ_EINVAL, "key d=%d and value d=%d differ", hk.hp.d, hv.hp.d);
    if (B < 0 || Hq < 0 || Hkv <= 0 || T_max < 0) return fail(TQ_EINVAL, "negative or zero shape");
    if (Hq % Hkv != 0) return fail(TQ_EINVAL, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
    const int G = Hq / Hkv;
    if (Hq > 4096) return fail(TQ_EUNSUPPORTED, "Hq=%d > 4096", Hq);
    if ((int64_t)B * Hkv * T_max > (int64_t)1 << 40) return fail(TQ_EINVAL, "cache too large");
    const int sms = hk.num_sms > 0 ? hk.num_sms : 148;
    DecodeShape p;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.T_max = T_max; p.d = hk.hp.d; p.G = G;
    const int hper = use_mma_split(p.d) ? mmadec::kHeadsPerCta : kMaxGroup;
    const int64_t units = (int64_t)(B > 0 ? B : 1) * Hkv * ((G + hper - 1) / hper);
    // CUDA-core path: two CTAs per SM; tensor-core path: one 16-warp CTA per SM,
    // and no more CTAs than SMs so that every split runs in the same wave.
    int64_t want = use_mma_split(p.d) ? (int64_t)sms * mmadec::ctas_per_sm(hv.hp.variant == TQ_PROD) / units
                                      : (2 * (int64_t)sms + units - 1) / units;
    int64_t max_splits = (T_max + kMinChunk - 1) / kMinChunk;
    if (max_splits < 1) max_splits = 1;
    if (use_mma_split(p.d) && want > mmadec::kMaxSplitsMerged) want = mmadec::kMaxSplitsMerged;
    if (want > max_splits) want = max_splits;
    if (want < 1) want = 1;
    int64_t chunk = (T_max + want - 1) / want;
    chunk = (chunk + kMinChunk - 1) / kMinChunk * kMinChunk;
    if (chunk < kMinChunk) chunk = kMinChunk;
    // Tensor-core path: a CTA takes at most kMaxChunk tokens, so that a batch of
    // ragged lengths (unknown on the host) is spread over several waves of CTAs
    // that the hardware hands out as SMs free up, instead of one CTA per slab
    // whose longest slab sets the time.  Equal-length workloads already fill one
    // wave with smaller chunks and are unaffected.
    if (use_mma_split(p.d) && chunk > kMaxChunk) {
        // … but never more splits than the last CTA of a group can merge
        const int64_t floor_chunk = ((T_max + mmadec::kMaxSplitsMerged - 1) / mmadec::kMaxSplitsMerged + kMinChunk - 1) /
                                    kMinChunk * kMinChunk;
        chunk = kMaxChunk > floor_chunk ? kMaxChunk : floor_chunk;
    }
    p.chunk = (int)chunk;
    p.n_splits = (int)((T_max + chunk - 1) / chunk);
    if (p.n_splits < 1) p.n_splits = 1;
    *plan = p;
    *ws_bytes = ws_layout(p, hv.hp.variant == TQ_PROD).total;
    return TQ_OK;
}

int64_t decode_split_ctas(const DecodeShape& plan) {
    const int hper = use_mma_split(plan.d) ? mmadec::kHeadsPerCta : kMaxGroup;
    return (int64_t)plan.n_splits * plan.Hkv * ((plan.G + hper - 1) / hper) * plan.B;
}

int* decode_tickets(const tq_ctx& hv, const DecodeShape& plan, void* workspace, int* count) {
    const WsLayout w = ws_layout(plan, hv.hp.variant == TQ_PROD);
    *count = plan.B * plan.Hq;
    return reinterpret_cast<int*>(static_cast<char*>(workspace) + w.cnt);
}

int launch_decode(const tq_ctx& hk, const tq_ctx& hv, const DecodeShape& plan, const void* q, int q_dtype,
                  const tq_planes& kc, const tq_planes& vc, const int32_t* seq_lens, float scale, float* out,
                  float* scores_out, void* workspace, cudaStream_t s, bool tickets_zeroed) {
    switch (plan.d) {
        case 32: return launch_d<32>(hk, hv, plan, q, q_dtype, kc, vc, seq_lens, scale, out, scores_out, workspace, s, tickets_zeroed);
        case 64: return launch_d<64>(hk, hv, plan, q, q_dtype, kc, vc, seq_lens, scale, out, scores_out, workspace, s, tickets_zeroed);
        case 96: return launch_d<96>(hk, hv, plan, q, q_dtype, kc, vc, seq_lens, scale, out, scores_out, workspace, s, tickets_zeroed);
        case 128: return launch_d<128>(hk, hv, plan, q, q_dtype, kc, vc, seq_lens, scale, out, scores_out, workspace, s, tickets_zeroed);
        case 160: return launch_d<160>(hk, hv, plan, q, q_dtype, kc, vc, seq_lens, scale, out, scores_out, workspace, s, tickets_zeroed);
        case 192: return launch_d<192>(hk, hv, plan, q, q_dtype, kc, vc, seq_lens, scale, out, scores_out, workspace, s, tickets_zeroed);
        case 224: return launch_d<224>(hk, hv, plan, q, q_dtype, kc, vc, seq_lens, scale, out, scores_out, workspace, s, tickets_zeroed);
        case 256: return launch_d<256>(hk, hv, plan, q, q_dtype, kc, vc, seq_lens, scale, out, scores_out, workspace, s, tickets_zeroed);
        default: return fail(TQ_EUNSUPPORTED, "d=%d", plan.d);
    }
}

}  // namespace tq
