// Outlier-channel mixed precision: every row's d channels split into d_o outlier
// channels and d − d_o others, each part quantized by its own TurboQuant handle
// (own norm, rotation and codebook; the page's experiments use 32 channels at 3
// bits and 96 at 2).  The split is a device permutation perm[d]: perm[0..d_o)
// are the outlier channels, perm[d_o..d) the rest.
//
// Here: choosing the outlier channels (largest energy over the rows to be
// cached), and split-K decode attention whose keys and values are two-part rows.
// A token's score is the sum of its parts' scores; values accumulate per part in
// that part's rotated frame and each part is rotated back and scattered to its
// channels once per output head.  Lane l of a warp owns positions j = l + 32m of
// the permuted row; d_o is a multiple of 32, so each slot m lies in one part.
#include <math.h>

#include "tq_common.cuh"
#include "tq_decode_args.h"
#include "tq_mixed_decode.h"

namespace tq {
namespace {

constexpr int kWarps = 4;      // warps per split CTA
// query heads per split CTA: their queries and value sums are held in registers
__host__ __device__ constexpr int heads_per_cta(int d) { return d <= 128 ? 8 : 4; }
constexpr int kMinChunk = 64;  // tokens per split at least

// ---------------------------------------------------------------- outlier channels
// energy[j] += Σ_rows x_j² over this block's rows, in double.
template <typename TIn>
__global__ void channel_energy_kernel(const TIn* __restrict__ x, int64_t n_rows, int64_t stride, int d,
                                      int64_t rows_per_block, double* __restrict__ energy) {
    const int j = threadIdx.x;
    const int64_t r0 = (int64_t)blockIdx.x * rows_per_block;
    const int64_t r1 = r0 + rows_per_block < n_rows ? r0 + rows_per_block : n_rows;
    if (j >= d) return;
    double e = 0.0;
    for (int64_t r = r0; r < r1; ++r) {
        const double v = load_elem(x + r * stride + j);
        e = fma(v, v, e);
    }
    atomicAdd(energy + j, e);
}

// One block of d threads: the d_o channels of largest energy (ties to the lower
// index) in ascending order, then the others in ascending order.
__global__ void outlier_perm_kernel(const double* __restrict__ energy, int d, int d_o, int32_t* __restrict__ perm) {
    __shared__ double e[kMaxD];
    __shared__ int is_out[kMaxD];
    const int j = threadIdx.x;
    if (j < d) e[j] = energy[j];
    __syncthreads();
    int rank = 0;
    if (j < d)
        for (int k = 0; k < d; ++k) rank += (e[k] > e[j] || (e[k] == e[j] && k < j)) ? 1 : 0;
    if (j < d) is_out[j] = rank < d_o;
    __syncthreads();
    if (j < d) {
        int before = 0;  // channels of the same class below j
        for (int k = 0; k < j; ++k) before += is_out[k] == is_out[j] ? 1 : 0;
        perm[is_out[j] ? before : d_o + before] = j;
    }
}

// ---------------------------------------------------------------- decode
// One part of a split row: its handle's tables and its planes.
struct Part {
    const uint8_t* codes;
    const uint8_t* signs;
    const float* norm;
    const float* rnorm;
    Codebook cb;
    int b;         // b_m
    int d;         // channels of the part
    float gamma;   // √(π/2)/d_part
};

struct MixedArgs {
    Part k[2], v[2];         // [0] outlier part, [1] the rest
    int kdo, vdo;            // d_o of the key and value splits
    const int32_t* seq_lens;
    const float* qr;         // [B·Hq][D] rotated query parts, key-permuted positions
    const float* qs;         // same for S·q (prod keys)
    float* pm;
    float* pl;
    float* pacc;
    float* pacc2;
    float* scores;
    float scale;
    int B, Hq, Hkv, T_max, G, n_splits, chunk, n_hblocks;
};

// q′ (and q″ for prod keys) of each key part: position j of part p is
// Σ_i Π_p[jl][i]·q[perm[off_p + i]] with jl = j − off_p.
template <int D, typename TQ>
__global__ void mixed_query_prep_kernel(const TQ* __restrict__ q, const int32_t* __restrict__ perm, int kdo,
                                        const float* __restrict__ PiT0, const float* __restrict__ ST0,
                                        const float* __restrict__ PiT1, const float* __restrict__ ST1, int kprod,
                                        int Hq, float* __restrict__ qr, float* __restrict__ qs, int* __restrict__ status) {
    __shared__ float qv[D];
    const int h = blockIdx.x, b = blockIdx.y, j = threadIdx.x;
    const size_t base = ((size_t)b * Hq + h) * D;
    ChannelMap cm;
    cm.ch = perm;
    cm.d_full = D;
    cm.status = status;
    qv[j] = load_elem(q + base + channel_of(cm, j));  // qv in key-permuted order
    __syncthreads();
    const bool p0 = j < kdo;
    const int off = p0 ? 0 : kdo, dp = p0 ? kdo : D - kdo, jl = j - off;
    const float* PiT = p0 ? PiT0 : PiT1;
    const float* ST = p0 ? ST0 : ST1;
    float a = 0.f, c = 0.f;
#pragma unroll 16
    for (int i = 0; i < dp; ++i) {  // unrolled so that the matrix loads go out in batches
        a = fmaf(__ldg(PiT + (size_t)i * dp + jl), qv[off + i], a);
        if (kprod) c = fmaf(__ldg(ST + (size_t)i * dp + jl), qv[off + i], c);
    }
    qr[base + j] = a;
    if (kprod) qs[base + j] = c;
}

// Split-K flash decoding over token chunks for two-part keys and values: per
// (token chunk, KV head, block of kHB query heads) an online softmax and per-part
// value sums, written as one partial (m, l, acc[, acc2]) per head.  The block's
// q′ (and for prod keys q″) and value sums live in registers; a group smaller
// than kHB pads with zero queries whose results are not written.
template <int D, bool KPROD, bool VPROD>
__global__ void __launch_bounds__(kWarps * 32, 2)
mixed_split_kernel(const MixedArgs a) {
    constexpr int PER = D / 32;
    constexpr int kHB = heads_per_cta(D);
    extern __shared__ float sm[];
    const int hb = blockIdx.y % a.n_hblocks, kvh = blockIdx.y / a.n_hblocks;
    const int G = min(kHB, a.G - hb * kHB);           // live heads of this block
    float* wacc = sm;                                 // [warps][kHB][D] value sums at the end
    float* acc2 = wacc + kWarps * kHB * D;            // [warps][kHB][D] (prod values)
    float* wm = acc2 + (VPROD ? kWarps * kHB * D : 0);  // [warps][kHB]
    float* wl = wm + kWarps * kHB;                    // [warps][kHB]
    __shared__ float cent[4][kMaxLevels];             // key part 0, 1, value part 0, 1

    const int split = blockIdx.x, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int L = a.seq_lens[b];
    L = L < 0 ? 0 : (L > a.T_max ? a.T_max : L);
    const int t0 = split * a.chunk;
    const int t1 = min(t0 + a.chunk, L);
    const size_t head0 = (size_t)b * a.Hq + (size_t)kvh * a.G + (size_t)hb * kHB;

    if (VPROD)
        for (int i = threadIdx.x; i < kWarps * kHB * D; i += blockDim.x) acc2[i] = 0.f;
    if (threadIdx.x < kMaxLevels) {
        const int i = threadIdx.x;
        cent[0][i] = a.k[0].cb.c[i];
        cent[1][i] = a.k[1].cb.c[i];
        cent[2][i] = a.v[0].cb.c[i];
        cent[3][i] = a.v[1].cb.c[i];
    }
    float q1[kHB][PER], q2[KPROD ? kHB : 1][PER], acc[kHB][PER], m_[kHB], l_[kHB];
#pragma unroll
    for (int h = 0; h < kHB; ++h) {
        m_[h] = -INFINITY;
        l_[h] = 0.f;
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            const bool live = h < G;
            q1[h][m] = live ? a.qr[(head0 + h) * D + lane + 32 * m] : 0.f;
            if (KPROD) q2[h][m] = live ? a.qs[(head0 + h) * D + lane + 32 * m] : 0.f;
            acc[h][m] = 0.f;
        }
    }
    __syncthreads();
    float* myacc2 = acc2 + warp * kHB * D;
    // record sizes of the four parts' planes
    const int kcb0 = a.k[0].b * a.k[0].d / 8, kcb1 = a.k[1].b * a.k[1].d / 8;
    const int vcb0 = a.v[0].b * a.v[0].d / 8, vcb1 = a.v[1].b * a.v[1].d / 8;

    // A token's raw words: for each slot the code word(s) holding its lane's code
    // and the sign word, for keys and values, and the parts' norms.  The next
    // token's are loaded while the current one is computed.
    uint32_t kw[PER][2], ks[PER], vw[PER][2], vs[PER];
    float nr[8];
    auto load_raw = [&](int64_t row) {
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            {
                const bool o = 32 * m < a.kdo;
                const int jl = lane + 32 * m - (o ? 0 : a.kdo);
                const int bp = o ? a.k[0].b : a.k[1].b;
                kw[m][0] = kw[m][1] = 0u;
                if (bp > 0) {
                    const uint32_t* w = reinterpret_cast<const uint32_t*>(o ? a.k[0].codes + row * kcb0
                                                                            : a.k[1].codes + row * kcb1);
                    const int bit = jl * bp;
                    kw[m][0] = w[bit >> 5];
                    if ((bit & 31) + bp > 32) kw[m][1] = w[(bit >> 5) + 1];
                }
                if (KPROD) {
                    const uint8_t* sp = o ? a.k[0].signs + row * (a.k[0].d / 8) : a.k[1].signs + row * (a.k[1].d / 8);
                    ks[m] = reinterpret_cast<const uint32_t*>(sp)[jl >> 5];
                }
            }
            {
                const bool o = 32 * m < a.vdo;
                const int jl = lane + 32 * m - (o ? 0 : a.vdo);
                const int bp = o ? a.v[0].b : a.v[1].b;
                vw[m][0] = vw[m][1] = 0u;
                if (bp > 0) {
                    const uint32_t* w = reinterpret_cast<const uint32_t*>(o ? a.v[0].codes + row * vcb0
                                                                            : a.v[1].codes + row * vcb1);
                    const int bit = jl * bp;
                    vw[m][0] = w[bit >> 5];
                    if ((bit & 31) + bp > 32) vw[m][1] = w[(bit >> 5) + 1];
                }
                if (VPROD) {
                    const uint8_t* sp = o ? a.v[0].signs + row * (a.v[0].d / 8) : a.v[1].signs + row * (a.v[1].d / 8);
                    vs[m] = reinterpret_cast<const uint32_t*>(sp)[jl >> 5];
                }
            }
        }
        nr[0] = a.k[0].norm[row];
        nr[1] = a.k[1].norm[row];
        nr[2] = a.v[0].norm[row];
        nr[3] = a.v[1].norm[row];
        nr[4] = KPROD ? a.k[0].rnorm[row] : 0.f;
        nr[5] = KPROD ? a.k[1].rnorm[row] : 0.f;
        nr[6] = VPROD ? a.v[0].rnorm[row] : 0.f;
        nr[7] = VPROD ? a.v[1].rnorm[row] : 0.f;
    };
    const int64_t slab = ((int64_t)b * a.Hkv + kvh) * a.T_max;
    if (t0 + warp < t1) load_raw(slab + t0 + warp);

    for (int t = t0 + warp; t < t1; t += kWarps) {
        float ck[PER], zk[PER], cv[PER], zv[PER];
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            {
                const bool o = 32 * m < a.kdo;
                const int jl = lane + 32 * m - (o ? 0 : a.kdo);
                const int bp = o ? a.k[0].b : a.k[1].b;
                const int code = (int)(__funnelshift_r(kw[m][0], kw[m][1], (jl * bp) & 31) & ((1u << bp) - 1u));
                ck[m] = bp > 0 ? cent[o ? 0 : 1][code] : 0.f;
                if (KPROD) zk[m] = ((ks[m] >> lane) & 1u) ? 1.f : -1.f;
            }
            {
                const bool o = 32 * m < a.vdo;
                const int jl = lane + 32 * m - (o ? 0 : a.vdo);
                const int bp = o ? a.v[0].b : a.v[1].b;
                const int code = (int)(__funnelshift_r(vw[m][0], vw[m][1], (jl * bp) & 31) & ((1u << bp) - 1u));
                cv[m] = bp > 0 ? cent[o ? 2 : 3][code] : 0.f;
                if (VPROD) zv[m] = ((vs[m] >> lane) & 1u) ? 1.f : -1.f;
            }
        }
        const float kn0 = nr[0], kn1 = nr[1], vn0 = nr[2], vn1 = nr[3];
        const float krn0 = a.k[0].gamma * nr[4], krn1 = a.k[1].gamma * nr[5];
        const float vrn0 = a.v[0].gamma * nr[6], vrn1 = a.v[1].gamma * nr[7];
        // the next token's words are in flight while this one is computed
        if (t + kWarps < t1) load_raw(slab + t + kWarps);
        // the key's per-slot factors: ‖k_p‖·c and ‖k_p‖·γ_p‖r_p‖·z
        float fk[PER], gk[PER];
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            const bool o = 32 * m < a.kdo;
            fk[m] = (o ? kn0 : kn1) * ck[m];
            if (KPROD) gk[m] = (o ? kn0 * krn0 : kn1 * krn1) * zk[m];
        }
        // every head's score: lane shares, then all heads reduced together
        float part[kHB];
#pragma unroll
        for (int h = 0; h < kHB; ++h) {
            float s = 0.f;
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                s = fmaf(q1[h][m], fk[m], s);
                if (KPROD) s = fmaf(q2[h][m], gk[m], s);
            }
            part[h] = s;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int h = 0; h < kHB; ++h) part[h] += __shfl_xor_sync(0xffffffffu, part[h], off);
        // the value's per-slot factors ‖v_p‖·c and ‖v_p‖·γ_p‖r_p‖·z
        float fv[PER], gv[PER];
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            const bool o = 32 * m < a.vdo;
            fv[m] = (o ? vn0 : vn1) * cv[m];
            if (VPROD) gv[m] = (o ? vn0 * vrn0 : vn1 * vrn1) * zv[m];
        }
#pragma unroll
        for (int h = 0; h < kHB; ++h) {
            const float s = a.scale * part[h];
            if (a.scores != nullptr && lane == 0 && h < G) a.scores[(head0 + h) * a.T_max + t] = s;
            // online softmax (all lanes hold identical values)
            const float mn = fmaxf(m_[h], s);
            const float corr = __expf(m_[h] - mn);
            const float p = __expf(s - mn);
            l_[h] = fmaf(l_[h], corr, p);
            m_[h] = mn;
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                acc[h][m] = fmaf(acc[h][m], corr, p * fv[m]);
                if (VPROD) {
                    float* r2 = myacc2 + h * D + lane + 32 * m;
                    *r2 = fmaf(*r2, corr, p * gv[m]);
                }
            }
        }
    }
#pragma unroll
    for (int h = 0; h < kHB; ++h) {
#pragma unroll
        for (int m = 0; m < PER; ++m) wacc[(warp * kHB + h) * D + lane + 32 * m] = acc[h][m];
        if (lane == 0) {
            wm[warp * kHB + h] = m_[h];
            wl[warp * kHB + h] = l_[h];
        }
    }
    __syncthreads();

    // combine the warps of this split and write its partial state (live heads only)
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
        const int h = i / D, j = i % D;
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * kHB + h]);
        float o = 0.f, o2 = 0.f, l = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < kWarps; ++w) {
                const float f = __expf(wm[w * kHB + h] - M);
                o = fmaf(f, wacc[(w * kHB + h) * D + j], o);
                if (VPROD) o2 = fmaf(f, acc2[(w * kHB + h) * D + j], o2);
                l = fmaf(f, wl[w * kHB + h], l);
            }
        }
        const size_t ps = (head0 + h) * a.n_splits + split;
        a.pacc[ps * D + j] = o;
        if (VPROD) a.pacc2[ps * D + j] = o2;
        if (j == 0) {
            a.pm[ps] = M;
            a.pl[ps] = l;
        }
    }
}

// Combine the splits of one head, rotate each value part back (out = Π_pᵀ·acc_p/l
// + S_pᵀ·acc2_p/l) and scatter it to its channels.
template <int D, bool VPROD>
__global__ void mixed_merge_kernel(const float* __restrict__ pm, const float* __restrict__ pl,
                                   const float* __restrict__ pacc, const float* __restrict__ pacc2,
                                   const float* __restrict__ Pi0, const float* __restrict__ S0,
                                   const float* __restrict__ Pi1, const float* __restrict__ S1, int vdo,
                                   const int32_t* __restrict__ perm_v, int Hq, int n_splits, float* __restrict__ out,
                                   int* __restrict__ status) {
    __shared__ float o1[D], o2[D];
    const int h = blockIdx.x, b = blockIdx.y, j = threadIdx.x;
    const size_t head = (size_t)b * Hq + h;
    float M = -INFINITY;
#pragma unroll 16
    for (int s = 0; s < n_splits; ++s) M = fmaxf(M, pm[head * n_splits + s]);
    float a = 0.f, c = 0.f, l = 0.f;
    if (M != -INFINITY) {
#pragma unroll 8
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
    const bool p0 = j < vdo;
    const int off = p0 ? 0 : vdo, dp = p0 ? vdo : D - vdo, jl = j - off;
    const float* Pi = p0 ? Pi0 : Pi1;
    const float* S = p0 ? S0 : S1;
    float r = 0.f;
#pragma unroll 16
    for (int k = 0; k < dp; ++k) {
        r = fmaf(__ldg(Pi + (size_t)k * dp + jl), o1[off + k], r);
        if (VPROD) r = fmaf(__ldg(S + (size_t)k * dp + jl), o2[off + k], r);
    }
    ChannelMap cm;
    cm.ch = perm_v;
    cm.d_full = D;
    cm.status = status;
    out[head * D + channel_of(cm, j)] = r;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct MixedLayout {
    size_t qr, qs, pm, pl, pacc, pacc2, cnt, total;
};

// The CUDA-core path keeps rotated queries (qr, qs) and separate merge
// partials for prod values; the tensor-core path needs split maxima, sums,
// value sums and one merge ticket per head (cnt).
MixedLayout mixed_layout(int B, int Hq, int d, int n_splits, bool vprod, bool tc = false) {
    MixedLayout w;
    const size_t heads = (size_t)B * Hq;
    size_t off = 0;
    w.qr = off;
    if (!tc) off = align256(off + heads * d * 4);
    w.qs = off;
    if (!tc) off = align256(off + heads * d * 4);
    w.pm = off;
    off = align256(off + heads * n_splits * 4);
    w.pl = off;
    off = align256(off + heads * n_splits * 4);
    w.pacc = off;
    off = align256(off + heads * n_splits * d * 4);
    w.pacc2 = off;
    if (vprod) off = align256(off + heads * n_splits * d * 4);
    w.cnt = off;
    if (tc) off = align256(off + heads * 4);
    w.total = off > 0 ? off : 256;
    return w;
}

int launch_mixed_tc_path(const MixedDecode& m, const MixedShape& p, cudaStream_t s) {
    const MixedLayout w = mixed_layout(p.B, p.Hq, p.d, p.n_splits, false, true);
    char* ws = static_cast<char*>(m.workspace);
    MixedTcArgs a;
    for (int i = 0; i < 2; ++i) {
        a.kc[i] = m.kc[i].codes;
        a.kn[i] = m.kc[i].norm;
        a.vc[i] = m.vc[i].codes;
        a.vn[i] = m.vc[i].norm;
        a.kcb[i] = m.hk[i]->cb;
        a.vcb[i] = m.hv[i]->cb;
        a.kPi_hi[i] = m.hk[i]->dp.Pi_hi;
        a.kPi_lo[i] = m.hk[i]->dp.Pi_lo;
        a.vPiT_hi[i] = m.hv[i]->dp.PiT_hi;
        a.vPiT_lo[i] = m.hv[i]->dp.PiT_lo;
        a.ks[i] = m.kc[i].signs;
        a.kr[i] = m.kc[i].rnorm;
        a.kS_hi[i] = m.hk[i]->dp.S_hi;
        a.kS_lo[i] = m.hk[i]->dp.S_lo;
        a.kgamma[i] = m.hk[i]->gamma;
    }
    a.kp = m.hk[0]->hp.variant == TQ_PROD;
    a.seq_lens = m.seq_lens;
    a.perm_k = m.perm_k;
    a.perm_v = m.perm_v;
    a.pm = reinterpret_cast<float*>(ws + w.pm);
    a.pl = reinterpret_cast<float*>(ws + w.pl);
    a.pacc = reinterpret_cast<float*>(ws + w.pacc);
    a.cnt = reinterpret_cast<int*>(ws + w.cnt);
    a.out = m.out;
    a.scores = m.scores;
    a.scale = m.scale;
    a.B = p.B; a.Hq = p.Hq; a.Hkv = p.Hkv; a.T_max = p.T_max; a.G = p.G;
    a.n_splits = p.n_splits; a.chunk = p.chunk;
    a.n_hblocks = (p.G + mmadec::kHeadsPerCta - 1) / mmadec::kHeadsPerCta;
    a.q = m.q;
    a.q_f32 = m.q_dtype == TQ_F32;
    a.status = m.hk[0]->dp.status;
    const int rc = launch_clear_tickets(a.cnt, p.B * p.Hq, s);
    if (rc != TQ_OK) return rc;
    return launch_mixed_decode_tc(a, dim3(p.n_splits, p.Hkv * a.n_hblocks, p.B), m.hk[0]->hp.b_mse,
                                  m.hk[1]->hp.b_mse, s);
}

void fill_part(Part* p, const tq_ctx& h, const tq_planes& pl) {
    p->codes = pl.codes;
    p->signs = pl.signs;
    p->norm = pl.norm;
    p->rnorm = pl.rnorm;
    p->cb = h.cb;
    p->b = h.hp.b_mse;
    p->d = h.hp.d;
    p->gamma = h.gamma;
}

template <int D>
int launch_mixed_d(const MixedDecode& m, const MixedShape& p, cudaStream_t s) {
    const bool kprod = m.hk[0]->hp.variant == TQ_PROD, vprod = m.hv[0]->hp.variant == TQ_PROD;
    const MixedLayout w = mixed_layout(p.B, p.Hq, D, p.n_splits, vprod);
    char* ws = static_cast<char*>(m.workspace);
    MixedArgs a;
    for (int i = 0; i < 2; ++i) {
        fill_part(&a.k[i], *m.hk[i], m.kc[i]);
        fill_part(&a.v[i], *m.hv[i], m.vc[i]);
    }
    a.kdo = m.hk[0]->hp.d;
    a.vdo = m.hv[0]->hp.d;
    a.seq_lens = m.seq_lens;
    float* qr = reinterpret_cast<float*>(ws + w.qr);
    float* qs = reinterpret_cast<float*>(ws + w.qs);
    a.qr = qr;
    a.qs = qs;
    a.pm = reinterpret_cast<float*>(ws + w.pm);
    a.pl = reinterpret_cast<float*>(ws + w.pl);
    a.pacc = reinterpret_cast<float*>(ws + w.pacc);
    a.pacc2 = reinterpret_cast<float*>(ws + w.pacc2);
    a.scores = m.scores;
    a.scale = m.scale;
    a.B = p.B; a.Hq = p.Hq; a.Hkv = p.Hkv; a.T_max = p.T_max; a.G = p.G;
    a.n_splits = p.n_splits; a.chunk = p.chunk;
    constexpr int kHB = heads_per_cta(D);
    a.n_hblocks = (p.G + kHB - 1) / kHB;
    int* status = m.hk[0]->dp.status;
    const dim3 pg(p.Hq, p.B);
    const tq_ctx& k0 = *m.hk[0];
    const tq_ctx& k1 = *m.hk[1];
    if (m.q_dtype == TQ_F32)
        mixed_query_prep_kernel<D, float><<<pg, D, 0, s>>>(static_cast<const float*>(m.q), m.perm_k, a.kdo, k0.dp.PiT,
                                                           k0.dp.ST, k1.dp.PiT, k1.dp.ST, kprod, p.Hq, qr, qs, status);
    else
        mixed_query_prep_kernel<D, __nv_bfloat16><<<pg, D, 0, s>>>(static_cast<const __nv_bfloat16*>(m.q), m.perm_k,
                                                                   a.kdo, k0.dp.PiT, k0.dp.ST, k1.dp.PiT, k1.dp.ST,
                                                                   kprod, p.Hq, qr, qs, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "mixed query prep launch");

    const size_t smem = sizeof(float) * ((size_t)kWarps * kHB * D * (vprod ? 2 : 1) + 2 * kWarps * kHB);
    const dim3 sg(p.n_splits, p.Hkv * a.n_hblocks, p.B);
#define TQ_MSPLIT(KP, VP)                                                                        \
    do {                                                                                         \
        auto fn = mixed_split_kernel<D, KP, VP>;                                                 \
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);   \
        if (e != cudaSuccess) return cuda_fail(e, "mixed decode smem attribute");               \
        fn<<<sg, kWarps * 32, smem, s>>>(a);                                                     \
    } while (0)
    if (kprod && vprod) TQ_MSPLIT(true, true);
    else if (kprod) TQ_MSPLIT(true, false);
    else if (vprod) TQ_MSPLIT(false, true);
    else TQ_MSPLIT(false, false);
#undef TQ_MSPLIT
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "mixed decode split launch");
    const tq_ctx& v0 = *m.hv[0];
    const tq_ctx& v1 = *m.hv[1];
    if (vprod)
        mixed_merge_kernel<D, true><<<pg, D, 0, s>>>(a.pm, a.pl, a.pacc, a.pacc2, v0.dp.Pi, v0.dp.S, v1.dp.Pi, v1.dp.S,
                                                     a.vdo, m.perm_v, p.Hq, p.n_splits, m.out, status);
    else
        mixed_merge_kernel<D, false><<<pg, D, 0, s>>>(a.pm, a.pl, a.pacc, a.pacc2, v0.dp.Pi, v0.dp.S, v1.dp.Pi,
                                                      v1.dp.S, a.vdo, m.perm_v, p.Hq, p.n_splits, m.out, status);
    e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "mixed decode merge launch");
}

}  // namespace

bool mixed_decode_tc_supported(const tq_ctx& hko, const tq_ctx& hkn, const tq_ctx& hvo, const tq_ctx& hvn,
                               int T_max) {
    const tq_ctx* hs[4] = {&hko, &hkn, &hvo, &hvn};
    for (const tq_ctx* h : hs)
        if (h->dp.Pi_hi == nullptr || h->dp.PiT_hi == nullptr) return false;
    // values mse; keys both mse, or both prod with their S in bf16 hi/lo
    const bool kp = hko.hp.variant == TQ_PROD;
    if (hvo.hp.variant != TQ_MSE || hvn.hp.variant != TQ_MSE || hkn.hp.variant != hko.hp.variant) return false;
    if (kp && (hko.dp.S_hi == nullptr || hkn.dp.S_hi == nullptr)) return false;
    return hko.hp.d == 32 && hkn.hp.d == 96 && hvo.hp.d == 32 && hvn.hp.d == 96 && T_max % 4 == 0 &&
           hko.num_sms > 0 && mixed_tc_bits_supported(hko.hp.b_mse, hkn.hp.b_mse, hvo.hp.b_mse, hvn.hp.b_mse, kp);
}

int mixed_plan(int d, int sms, bool vprod, bool tc, int B, int Hq, int Hkv, int T_max, MixedShape* plan,
               size_t* ws_bytes) {
    if (B < 0 || Hq < 0 || Hkv <= 0 || T_max < 0) return fail(TQ_EINVAL, "negative or zero shape");
    if (Hq % Hkv != 0) return fail(TQ_EINVAL, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
    if (Hq > 4096) return fail(TQ_EUNSUPPORTED, "Hq=%d > 4096", Hq);
    if ((int64_t)B * Hkv * T_max > (int64_t)1 << 40) return fail(TQ_EINVAL, "cache too large");
    MixedShape p;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.T_max = T_max; p.d = d; p.G = Hq / Hkv;
    p.tc = tc;
    const int hb = tc ? mmadec::kHeadsPerCta : heads_per_cta(d);
    const int64_t units = (int64_t)(B > 0 ? B : 1) * Hkv * ((p.G + hb - 1) / hb);
    const int64_t nsm = sms > 0 ? sms : 148;
    // CUDA-core path: two waves of two resident 4-warp CTAs per SM; tensor-core
    // path: one CTA per SM in one wave, at most kMaxChunk tokens per CTA and no
    // more splits than the last CTA of a group merges
    int64_t want = tc ? nsm / units : (4 * nsm + units - 1) / units;
    int64_t max_splits = (T_max + kMinChunk - 1) / kMinChunk;
    if (max_splits < 1) max_splits = 1;
    if (tc && want > mmadec::kMaxSplitsMerged) want = mmadec::kMaxSplitsMerged;
    if (want > max_splits) want = max_splits;
    if (want < 1) want = 1;
    int64_t chunk = (T_max + want - 1) / want;
    chunk = (chunk + kMinChunk - 1) / kMinChunk * kMinChunk;
    if (chunk < kMinChunk) chunk = kMinChunk;
    constexpr int64_t kMaxChunkTc = 8192;
    if (tc && chunk > kMaxChunkTc) {
        const int64_t floor_chunk =
            ((T_max + mmadec::kMaxSplitsMerged - 1) / mmadec::kMaxSplitsMerged + kMinChunk - 1) / kMinChunk * kMinChunk;
        chunk = kMaxChunkTc > floor_chunk ? kMaxChunkTc : floor_chunk;
    }
    p.chunk = (int)chunk;
    p.n_splits = (int)((T_max + chunk - 1) / chunk);
    if (p.n_splits < 1) p.n_splits = 1;
    *plan = p;
    *ws_bytes = mixed_layout(B, Hq, d, p.n_splits, vprod, tc).total;
    return TQ_OK;
}

int launch_mixed_decode(const MixedDecode& m, const MixedShape& p, cudaStream_t s) {
    if (p.tc) return launch_mixed_tc_path(m, p, s);
    switch (p.d) {
        case 64: return launch_mixed_d<64>(m, p, s);
        case 96: return launch_mixed_d<96>(m, p, s);
        case 128: return launch_mixed_d<128>(m, p, s);
        case 160: return launch_mixed_d<160>(m, p, s);
        case 192: return launch_mixed_d<192>(m, p, s);
        case 224: return launch_mixed_d<224>(m, p, s);
        case 256: return launch_mixed_d<256>(m, p, s);
        default: return fail(TQ_EUNSUPPORTED, "mixed d=%d", p.d);
    }
}

int launch_select_outlier_channels(const void* x, int x_dtype, int64_t n_rows, int64_t stride, int d, int d_o,
                                   double* energy, int32_t* perm, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(energy, 0, (size_t)d * sizeof(double), s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the channel energies");
    if (n_rows > 0) {
        const int64_t per = 256;
        int64_t blocks = (n_rows + per - 1) / per;
        if (blocks > 0x7fffffffLL) return fail(TQ_EINVAL, "n_rows too large");
        if (x_dtype == TQ_F32)
            channel_energy_kernel<float><<<(unsigned)blocks, d, 0, s>>>(static_cast<const float*>(x), n_rows, stride,
                                                                         d, per, energy);
        else
            channel_energy_kernel<__nv_bfloat16><<<(unsigned)blocks, d, 0, s>>>(
                static_cast<const __nv_bfloat16*>(x), n_rows, stride, d, per, energy);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "channel energy launch");
    }
    outlier_perm_kernel<<<1, d, 0, s>>>(energy, d, d_o, perm);
    e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "outlier channel launch");
}

}  // namespace tq
