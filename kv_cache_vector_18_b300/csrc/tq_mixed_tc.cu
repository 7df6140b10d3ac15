// Outlier-channel mixed precision on the 5th-generation tensor cores (bf16 rows,
// mse parts, d = 128).
//
// Both parts of a row come out of one rotation: with P the channel permutation
// (outlier channels first), M = blockdiag(Π_o, Π_n)·P is orthogonal, and
// Y = X·Mᵀ holds the outlier part's rotated coordinates in its first d_o columns
// and the other part's in the rest.  M's bf16 hi/lo halves are the two handles'
// own Π_hi/Π_lo scattered through the permutation on the device (exact, and
// capturable in a CUDA graph), so the pipeline is the mse kernel's: a TMA
// producer warp, one thread issuing tcgen05.mma (hi then lo) into one of three
// TMEM accumulators, three epilogue warpgroups.  The epilogue differs: it keeps
// one norm per part, bucketizes each part's columns against that part's codebook
// and writes each part's codes and norm to that part's planes.  The keys and
// values of one step can share a launch: the grid's CTAs are divided between
// two parameter blocks (each with its own operand M, rows and planes).
#include "tq_common.cuh"
#include "tq_sm100.cuh"

namespace tq {
namespace {

using namespace sm100;

__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t x, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

constexpr int kD = 128;           // channels per row
constexpr int kTile = 128;        // rows per tile (MMA M)
constexpr int kKC = 64;           // K elements per 128-byte swizzle chunk
constexpr int kAcc = 3;           // TMEM accumulators = epilogue warpgroups
constexpr int kThreads = 32 * (2 + 4 * kAcc);
constexpr int kChunks = kD / kKC;
constexpr int kStageBytes = kTile * kD * 2;
constexpr int kChunkBytesA = kTile * 128;
constexpr int kChunkBytesB = kD * 128;
constexpr int kMatBytes = kD * kD * 2;
constexpr int kStages = 4;
constexpr uint32_t kTmemCols = 512;  // ≥ kAcc·kD
constexpr size_t kBarOffset = 2 * (size_t)kMatBytes + (size_t)kStages * kStageBytes;
constexpr size_t kSmemBytes = kBarOffset + 256 + 1024;

// M_hi / M_lo [j][c]: row j < d_o is row j of Π_o placed at the outlier
// channels, row j ≥ d_o row j − d_o of Π_n at the other channels, zero elsewhere.
struct OperandSrc {
    const uint16_t *po_hi, *po_lo, *pn_hi, *pn_lo;
    const int32_t* perm;
    int d_o;
    uint16_t *m_hi, *m_lo;
    int *status_o, *status_n;
};

// blockIdx.y picks the side (a single side launches one row of blocks).
__global__ void build_mixed_operand_kernel(const OperandSrc src_a, const OperandSrc src_b) {
    const OperandSrc& sr = blockIdx.y == 0 ? src_a : src_b;
    const uint16_t *po_hi = sr.po_hi, *po_lo = sr.po_lo, *pn_hi = sr.pn_hi, *pn_lo = sr.pn_lo;
    const int32_t* perm = sr.perm;
    const int d_o = sr.d_o;
    uint16_t *m_hi = sr.m_hi, *m_lo = sr.m_lo;
    int *status_o = sr.status_o, *status_n = sr.status_n;
    const int j = blockIdx.x, c = threadIdx.x;
    m_hi[(size_t)j * kD + c] = 0;
    m_lo[(size_t)j * kD + c] = 0;
    __syncthreads();
    const bool o = j < d_o;
    const int dp = o ? d_o : kD - d_o, jl = o ? j : j - d_o, off = o ? 0 : d_o;
    if (c < dp) {
        ChannelMap cm;
        cm.ch = perm + off;
        cm.d_full = kD;
        cm.status = o ? status_o : status_n;
        const int ch = channel_of(cm, c);
        m_hi[(size_t)j * kD + ch] = (o ? po_hi : pn_hi)[(size_t)jl * dp + c];
        m_lo[(size_t)j * kD + ch] = (o ? po_lo : pn_lo)[(size_t)jl * dp + c];
    }
}

// Codes of one 32-column chunk of a row against one part's boundaries: the mse
// kernel's arithmetic (saturated boundary tests, sign by bit operation, exact
// float packing), BM words out.
template <int BM>
__device__ __forceinline__ void bucket_chunk(const uint32_t* rc, uint64_t cs2, const float* kt2, uint32_t (&cw)[BM]) {
    constexpr int P = (1 << BM) / 2 - 1;
    constexpr int GB = BM == 3 ? 24 : 16;
    constexpr int GC = GB / BM;
    constexpr int NG = 32 / GC;
    constexpr float kAcc0 = (float)(1u << (GB - 1)) - 0.5f;
    uint64_t acc[NG];
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) acc[gi] = f2(kAcc0, 0.f);
#pragma unroll
    for (int k = 0; k < 32; k += 2) {
        const float va = __uint_as_float(rc[k]), vb = __uint_as_float(rc[k + 1]);
        uint64_t cnt2 = f2(0.5f, 0.5f);
        if constexpr (P > 0) {
            float wa, wb;
            f2_split(mul2(f2(va, vb), cs2), wa, wb);
#pragma unroll
            for (int p = 0; p < P; ++p)
                cnt2 = add2(cnt2, f2(__saturatef(fmaf(va, wa, kt2[p])), __saturatef(fmaf(vb, wb, kt2[p]))));
        }
        float ca, cb;
        f2_split(cnt2, ca, cb);
        const float sa = __uint_as_float(__float_as_uint(ca) | (__float_as_uint(va) & 0x80000000u));
        const float sb = __uint_as_float(__float_as_uint(cb) | (__float_as_uint(vb) & 0x80000000u));
        acc[k / GC] = fma2(f2(sa, sb), f2((float)(1u << (BM * (k % GC))), (float)(1u << (BM * ((k + 1) % GC)))),
                           acc[k / GC]);
    }
#pragma unroll
    for (int w = 0; w < BM; ++w) cw[w] = 0u;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        float ea, eb;
        f2_split(acc[gi], ea, eb);
        const uint32_t gbits = __float2uint_rn(ea + eb);
        const int bit = gi * GB, w = bit >> 5, sh = bit & 31;
        cw[w] |= gbits << sh;
        if (sh + GB > 32) cw[w + 1] |= gbits >> (32 - sh);
    }
}

template <int BM>
__device__ __forceinline__ void store_words(uint8_t* cd, const uint32_t (&cw)[BM], uint32_t keep) {
    if constexpr (BM == 4) {
        *reinterpret_cast<uint4*>(cd) = make_uint4(cw[0] & keep, cw[1] & keep, cw[2] & keep, cw[3] & keep);
    } else if constexpr (BM == 2) {
        *reinterpret_cast<uint2*>(cd) = make_uint2(cw[0] & keep, cw[1] & keep);
    } else {
#pragma unroll
        for (int w = 0; w < BM; ++w) reinterpret_cast<uint32_t*>(cd)[w] = cw[w] & keep;
    }
}

// Everything one side of a launch reads and writes: its rows (tm_x), its operand
// M (tm_m_hi, tm_m_lo), both parts' codebooks and planes, its status word.
struct MixSide {
    CUtensorMap tm_x, tm_m_hi, tm_m_lo;
    int64_t n_rows;
    Codebook cbo, cbn;
    uint8_t* codes_o;
    float* norm_o;
    uint8_t* codes_n;
    float* norm_n;
    int* status;
};

// CTAs [0, split) quantize side a, CTAs [split, gridDim.x) side b; a single side
// passes split = gridDim.x.
template <int DO, int BMO, int BMN>
__global__ void __launch_bounds__(kThreads, 1)
quantize_mixed_tc_kernel(const __grid_constant__ MixSide side_a, const __grid_constant__ MixSide side_b, int split) {
    const bool on_b = (int)blockIdx.x >= split;
    const MixSide& sd = on_b ? side_b : side_a;
    const int cta = on_b ? (int)blockIdx.x - split : (int)blockIdx.x;
    const int ncta = on_b ? (int)gridDim.x - split : split;
    const CUtensorMap& tm_x = sd.tm_x;
    const CUtensorMap& tm_m_hi = sd.tm_m_hi;
    const CUtensorMap& tm_m_lo = sd.tm_m_lo;
    const int64_t n_rows = sd.n_rows;
    const Codebook& cbo = sd.cbo;
    const Codebook& cbn = sd.cbn;
    uint8_t* __restrict__ codes_o = sd.codes_o;
    float* __restrict__ norm_o = sd.norm_o;
    uint8_t* __restrict__ codes_n = sd.codes_n;
    float* __restrict__ norm_n = sd.norm_n;
    int* __restrict__ status = sd.status;
    constexpr int DN = kD - DO;
    constexpr int CO = DO / 32;                       // 32-column chunks of the outlier part
    constexpr int PO = (1 << BMO) / 2 - 1, PN = (1 << BMN) / 2 - 1;
    constexpr int RO = BMO * DO / 8, RN = BMN * DN / 8;  // record bytes of the two code planes
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    allow_dependents();
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* m_hi = smem;
    uint8_t* m_lo = smem + kMatBytes;
    uint8_t* stages = smem + 2 * kMatBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOffset);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + kAcc;
    uint64_t* mat_full = tempty + kAcc;
    uint64_t* drain = mat_full + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = (n_rows + kTile - 1) / kTile;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(mat_full, 1);
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_holder, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ producer
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_m_hi);
        prefetch_tensormap(&tm_m_lo);
        mbar_arrive_expect_tx(mat_full, 2 * kMatBytes);
        for (int c = 0; c < kChunks; ++c) {
            tma_load_2d(m_hi + c * kChunkBytesB, &tm_m_hi, mat_full, c * kKC, 0);
            tma_load_2d(m_lo + c * kChunkBytesB, &tm_m_lo, mat_full, c * kKC, 0);
        }
        int64_t i = 0;
        for (int64_t tile = cta; tile < ntiles; tile += ncta, ++i) {
            const int s = (int)(i % kStages);
            const int64_t u = i / kStages;
            if (u > 0 && !mbar_wait(&empty[s], (uint32_t)((u - 1) & 1), status, 21)) break;
            mbar_arrive_expect_tx(&full[s], kStageBytes);
            uint8_t* st = stages + (size_t)s * kStageBytes;
            for (int c = 0; c < kChunks; ++c)
                tma_load_2d(st + c * kChunkBytesA, &tm_x, &full[s], c * kKC, (int)(tile * kTile));
        }
        // every load issued must have landed before the CTA may exit
        const int64_t issued = i;
        for (int64_t k = (issued > kStages ? issued - kStages : 0); k < issued; ++k)
            mbar_wait(&full[k % kStages], (uint32_t)((k / kStages) & 1), status, 22);
        mbar_wait(mat_full, 0, status, 22);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(kTile, kD);
        bool ok = mbar_wait(mat_full, 0, status, 23);
        tc_fence_after();
        const uint32_t a_base = smem_u32(stages), hi_base = smem_u32(m_hi), lo_base = smem_u32(m_lo);
        int64_t i = 0;
        for (int64_t tile = cta; ok && tile < ntiles; tile += ncta, ++i) {
            const int s = (int)(i % kStages);
            const int acc = (int)(i % kAcc);
            const int64_t ua = i / kAcc;
            if (!(ok = mbar_wait(&full[s], (uint32_t)((i / kStages) & 1), status, 24))) break;
            if (ua > 0 && !(ok = mbar_wait(&tempty[acc], (uint32_t)((ua - 1) & 1), status, 25))) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kD);
            const uint32_t a_stage = a_base + (uint32_t)(s * kStageBytes);
#pragma unroll
            for (int pass = 0; pass < 2; ++pass) {
                const uint32_t b_base = pass == 0 ? hi_base : lo_base;
#pragma unroll
                for (int c = 0; c < kChunks; ++c)
#pragma unroll
                    for (int kk = 0; kk < kKC / 16; ++kk) {
                        const uint64_t ad = smem_desc(a_stage + c * kChunkBytesA + kk * 32, 1024, 2);
                        const uint64_t bd = smem_desc(b_base + c * kChunkBytesB + kk * 32, 1024, 2);
                        mma_f16_ss(d_tmem, ad, bd, idesc, (pass | c | kk) != 0);
                    }
            }
            mma_commit(&empty[s]);
            mma_commit(&tfull[acc]);
        }
        mma_commit(drain);
        mbar_wait(drain, 0, status, 26);
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue
        const int wg = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int r_local = quad * 32 + lane;
        const int LO = 1 << BMO, LN = 1 << BMN;
        float t2o[PO > 0 ? PO : 1], t2n[PN > 0 ? PN : 1];  // squared positive boundaries
#pragma unroll
        for (int p = 0; p < PO; ++p) t2o[p] = cbo.t[LO / 2 + p] * cbo.t[LO / 2 + p];
#pragma unroll
        for (int p = 0; p < PN; ++p) t2n[p] = cbn.t[LN / 2 + p] * cbn.t[LN / 2 + p];
        const uint32_t taddr0 = tmem_base + (uint32_t)(wg * kD) + ((uint32_t)(quad * 32) << 16);
        int64_t j = 0;
        for (int64_t tile = cta + (int64_t)wg * ncta; tile < ntiles; tile += (int64_t)kAcc * ncta, ++j) {
            if (!mbar_wait(&tfull[wg], (uint32_t)(j & 1), status, 27)) break;
            tc_fence_after();
            // pass 1: ‖y_o‖² and ‖y_n‖² (the chunk index fixes the part at compile time)
            uint32_t r[2][32];
            uint64_t sso2 = 0ull, ssn2 = 0ull;
#pragma unroll
            for (int c = 0; c < kD / 32; c += 2) {
                tmem_ld32(taddr0 + c * 32, r[0]);
                tmem_ld32(taddr0 + (c + 1) * 32, r[1]);
                tmem_wait_ld(r[0]);
                tmem_wait_ld(r[1]);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int k = 0; k < 32; k += 2) {
                        const uint64_t v2 = f2(__uint_as_float(r[h][k]), __uint_as_float(r[h][k + 1]));
                        if (c + h < CO)
                            sso2 = fma2(v2, v2, sso2);
                        else
                            ssn2 = fma2(v2, v2, ssn2);
                    }
            }
            float sa, sb;
            f2_split(sso2, sa, sb);
            const float sso = sa + sb;
            f2_split(ssn2, sa, sb);
            const float ssn = sa + sb;
            const float no = sqrtf(sso), nn = sqrtf(ssn);
            // per part: c = K/‖y_p‖² (K = 2^62) and −K·t_p²
            const float cso = sso >= 0x1p-38f ? __fdividef(0x1p62f, sso) : 0x1p100f;
            const float csn = ssn >= 0x1p-38f ? __fdividef(0x1p62f, ssn) : 0x1p100f;
            const uint64_t cso2 = f2(cso, cso), csn2 = f2(csn, csn);
            float kto[PO > 0 ? PO : 1], ktn[PN > 0 ? PN : 1];
#pragma unroll
            for (int p = 0; p < PO; ++p) kto[p] = -(cso * sso) * t2o[p];
#pragma unroll
            for (int p = 0; p < PN; ++p) ktn[p] = -(csn * ssn) * t2n[p];
            const int64_t row = tile * kTile + r_local;
            const bool live = row < n_rows;
            const uint32_t keepo = no == 0.f ? 0u : 0xffffffffu, keepn = nn == 0.f ? 0u : 0xffffffffu;
            // pass 2: chunk c + 1 is loaded while chunk c is bucketized
            tmem_ld32(taddr0, r[0]);
#pragma unroll
            for (int c = 0; c < kD / 32; ++c) {
                tmem_wait_ld(r[c & 1]);
                if (c + 1 < kD / 32) tmem_ld32(taddr0 + (c + 1) * 32, r[(c + 1) & 1]);
                if (c < CO) {
                    uint32_t cw[BMO];
                    bucket_chunk<BMO>(r[c & 1], cso2, kto, cw);
                    if (live) store_words<BMO>(codes_o + row * (int64_t)RO + c * (BMO * 4), cw, keepo);
                } else {
                    uint32_t cw[BMN];
                    bucket_chunk<BMN>(r[c & 1], csn2, ktn, cw);
                    if (live) store_words<BMN>(codes_n + row * (int64_t)RN + (c - CO) * (BMN * 4), cw, keepn);
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[wg]);
            if (live) {
                norm_o[row] = no;
                norm_n[row] = nn;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// One launch over one side, or over two (b != nullptr, both holding rows): the
// grid's CTAs are divided between the sides in proportion to their tiles.
template <int DO, int BMO, int BMN>
int launch_mixed_tc(const MixSide& a, const MixSide* b, int num_sms, cudaStream_t s) {
    auto fn = quantize_mixed_tc_kernel<DO, BMO, BMN>;
    static std::atomic<uint64_t> smem_set{0};
    const int rc = ensure_smem_attr(smem_set, (const void*)fn, (int)kSmemBytes, "mixed quantize smem attribute");
    if (rc != TQ_OK) return rc;
    const int64_t ta = (a.n_rows + kTile - 1) / kTile;
    const int64_t tb = b ? (b->n_rows + kTile - 1) / kTile : 0;
    const int64_t tiles = ta + tb;
    const int grid = (int)(tiles < num_sms ? tiles : num_sms);
    int split = grid;
    if (b) {  // both sides hold ≥ 1 tile, so grid ≥ 2
        const int64_t want = (ta * grid + tiles / 2) / tiles;
        split = (int)(want < 1 ? 1 : (want > grid - 1 ? grid - 1 : want));
    }
    fn<<<grid, kThreads, kSmemBytes, s>>>(a, b ? *b : a, split);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "mixed tensor-core quantize launch");
}

template <int DO>
int dispatch_bits(int bo, int bn, const MixSide& a, const MixSide* b, int num_sms, cudaStream_t s) {
#define TQ_MB(BO, BN) \
    if (bo == BO && bn == BN) return launch_mixed_tc<DO, BO, BN>(a, b, num_sms, s)
    TQ_MB(1, 1); TQ_MB(2, 1); TQ_MB(2, 2); TQ_MB(3, 1); TQ_MB(3, 2);
    TQ_MB(3, 3); TQ_MB(4, 1); TQ_MB(4, 2); TQ_MB(4, 3); TQ_MB(4, 4);
#undef TQ_MB
    return fail(TQ_EUNSUPPORTED, "mixed tensor-core quantize: bits %d/%d", bo, bn);
}

// The operand source of one side, its M halves at scratch (2·kMatBytes).
OperandSrc operand_src(const tq_ctx& ho, const tq_ctx& hn, const int32_t* perm, void* scratch) {
    OperandSrc o;
    o.po_hi = ho.dp.Pi_hi;
    o.po_lo = ho.dp.Pi_lo;
    o.pn_hi = hn.dp.Pi_hi;
    o.pn_lo = hn.dp.Pi_lo;
    o.perm = perm;
    o.d_o = ho.hp.d;
    o.m_hi = static_cast<uint16_t*>(scratch);
    o.m_lo = o.m_hi + kD * kD;
    o.status_o = ho.dp.status;
    o.status_n = hn.dp.status;
    return o;
}

int make_mix_side(const tq_ctx& ho, const tq_ctx& hn, const OperandSrc& src, const void* x, int64_t n_rows,
                  int64_t stride, const tq_planes& out_o, const tq_planes& out_n, MixSide* sd) {
    int rc = encode_tmap_bf16_2d(&sd->tm_x, x, (uint64_t)kD, (uint64_t)n_rows, (uint64_t)stride * 2, kKC, kTile);
    if (rc == TQ_OK) rc = encode_tmap_bf16_2d(&sd->tm_m_hi, src.m_hi, kD, kD, (uint64_t)kD * 2, kKC, kD);
    if (rc == TQ_OK) rc = encode_tmap_bf16_2d(&sd->tm_m_lo, src.m_lo, kD, kD, (uint64_t)kD * 2, kKC, kD);
    sd->n_rows = n_rows;
    sd->cbo = ho.cb;
    sd->cbn = hn.cb;
    sd->codes_o = out_o.codes;
    sd->norm_o = out_o.norm;
    sd->codes_n = out_n.codes;
    sd->norm_n = out_n.norm;
    sd->status = ho.dp.status;
    return rc;
}

int launch_operands(const OperandSrc& a, const OperandSrc* b, cudaStream_t s) {
    build_mixed_operand_kernel<<<dim3(kD, b ? 2 : 1), kD, 0, s>>>(a, b ? *b : a);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "mixed operand launch");
}

}  // namespace

size_t mixed_tc_scratch_bytes() { return 2 * (size_t)kMatBytes; }

bool mixed_quantize_tc_supported(const tq_ctx& ho, const tq_ctx& hn, int x_dtype, int64_t n_rows, int64_t stride,
                                 const void* scratch, size_t scratch_bytes) {
    const int d_o = ho.hp.d, bo = ho.hp.b_mse, bn = hn.hp.b_mse;
    return x_dtype == TQ_BF16 && ho.hp.variant == TQ_MSE && d_o + hn.hp.d == kD && (d_o == 32 || d_o == 64) &&
           bn >= 1 && bn <= bo && bo <= 4 && ho.dp.Pi_hi != nullptr && hn.dp.Pi_hi != nullptr &&
           scratch != nullptr && scratch_bytes >= mixed_tc_scratch_bytes() &&
           (reinterpret_cast<uintptr_t>(scratch) & 255) == 0 && ((stride * 2) % 16) == 0 && ho.num_sms > 0 &&
           n_rows > 0 && n_rows < ((int64_t)1 << 31) - kTile;
}

int launch_mixed_quantize_tc(const tq_ctx& ho, const tq_ctx& hn, const int32_t* perm, const void* x, int64_t n_rows,
                             int64_t stride, const tq_planes& out_o, const tq_planes& out_n, void* scratch,
                             cudaStream_t s) {
    const OperandSrc src = operand_src(ho, hn, perm, scratch);
    int rc = launch_operands(src, nullptr, s);
    MixSide a;
    if (rc == TQ_OK) rc = make_mix_side(ho, hn, src, x, n_rows, stride, out_o, out_n, &a);
    if (rc != TQ_OK) return rc;
    if (ho.hp.d == 32) return dispatch_bits<32>(ho.hp.b_mse, hn.hp.b_mse, a, nullptr, ho.num_sms, s);
    return dispatch_bits<64>(ho.hp.b_mse, hn.hp.b_mse, a, nullptr, ho.num_sms, s);
}

bool mixed_quantize_pair_tc_supported(const tq_ctx& hko, const tq_ctx& hkn, const tq_ctx& hvo, const tq_ctx& hvn,
                                      int x_dtype, int64_t k_rows, int64_t k_stride, int64_t v_rows,
                                      int64_t v_stride, const void* scratch, size_t scratch_bytes) {
    return mixed_quantize_tc_supported(hko, hkn, x_dtype, k_rows, k_stride, scratch, scratch_bytes) &&
           mixed_quantize_tc_supported(hvo, hvn, x_dtype, v_rows, v_stride, scratch, scratch_bytes) &&
           scratch_bytes >= 2 * mixed_tc_scratch_bytes() && hko.hp.d == hvo.hp.d &&
           hko.hp.b_mse == hvo.hp.b_mse && hkn.hp.b_mse == hvn.hp.b_mse && hko.num_sms == hvo.num_sms;
}

int launch_mixed_quantize_pair_tc(const tq_ctx& hko, const tq_ctx& hkn, const tq_ctx& hvo, const tq_ctx& hvn,
                                  const int32_t* perm_k, const int32_t* perm_v, const void* k, const void* v,
                                  int64_t k_rows, int64_t k_stride, int64_t v_rows, int64_t v_stride,
                                  const tq_planes& k_out_o, const tq_planes& k_out_n, const tq_planes& v_out_o,
                                  const tq_planes& v_out_n, void* scratch, cudaStream_t s) {
    const OperandSrc sk = operand_src(hko, hkn, perm_k, scratch);
    const OperandSrc sv = operand_src(hvo, hvn, perm_v, static_cast<uint8_t*>(scratch) + mixed_tc_scratch_bytes());
    int rc = launch_operands(sk, &sv, s);
    MixSide a, b;
    if (rc == TQ_OK) rc = make_mix_side(hko, hkn, sk, k, k_rows, k_stride, k_out_o, k_out_n, &a);
    if (rc == TQ_OK) rc = make_mix_side(hvo, hvn, sv, v, v_rows, v_stride, v_out_o, v_out_n, &b);
    if (rc != TQ_OK) return rc;
    if (hko.hp.d == 32) return dispatch_bits<32>(hko.hp.b_mse, hkn.hp.b_mse, a, &b, hko.num_sms, s);
    return dispatch_bits<64>(hko.hp.b_mse, hkn.hp.b_mse, a, &b, hko.num_sms, s);
}

}  // namespace tq
