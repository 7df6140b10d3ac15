// tq_quantize on the 5th-generation tensor cores (tcgen05 + TMA + TMEM), for
// bf16 rows and the mse variant («Шаг 0»–«Шаг 2»).
//
// Per 128-row tile: Y = X·Πᵀ as two bf16 MMAs into one fp32 TMEM accumulator,
// Π = Π_hi + Π_lo (Π_hi = bf16(Π), Π_lo = bf16(Π − Π_hi)), so the rotation is
// accurate to ~2⁻¹⁷ relative while the inputs stay exact bf16.  With the
// Walsh–Hadamard rotation the operand is √d·Π = H·diag(σ), whose ±1 entries are
// exact in bf16: one MMA gives √d·y exactly up to fp32 accumulation, the
// codes depend only on y/‖y‖, and the stored norm is scaled by 1/√d.  The epilogue
// reads the accumulator row per thread, takes ‖y‖ = ‖x‖ (Π orthogonal), counts
// the norm-scaled Lloyd–Max boundaries below each y_j and packs b-bit codes.
//
// Epilogue arithmetic runs on the FP32 pipe, two coordinates per packed f32x2
// instruction where the operation allows it: with c = K/‖y‖² (K = 2^62), the
// test |y_j| > ‖y‖·t_p is the saturated step sat(y_j·(c·y_j) − K·t_p²) ∈ {0, 1}
// (one FFMA.SAT each; the exact product makes fractional values need a relative
// tie below 1e-16), the code is (L/2 − ½) ± (count + ½) with the sign of y_j put
// in by one bit operation, and codes are packed by exact float FMAs
// acc += code·2^(b·i), 16 or 24 bits per accumulator.
//
// Persistent CTAs (one per SM) with warp roles:
//   warp 0      TMA producer: Π_hi/Π_lo once, then X tiles into a STAGES ring
//   warp 1      TMEM owner and single-thread MMA issuer (three accumulators)
//   warps 2..13 three epilogue warpgroups, one per TMEM accumulator
#include "tq_common.cuh"
#include "tq_sm100.cuh"

namespace tq {
namespace {

using namespace sm100;

// Packed FP32 pair arithmetic (two lanes per instruction on the FP32 pipe).
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

constexpr int kTile = 128;        // rows per tile (MMA M)
constexpr int kKC = 64;           // K elements per 128-byte swizzle chunk
constexpr int kThreads = 32 * 14;  // 14 warps: 128 registers each

// F32: fp32 rows.  Four converter warps then load the rows with 16-byte loads and
// write each value as bf16 hi + lo into two swizzled tiles (x = x_hi + x_lo to
// ~2⁻¹⁸), and the MMAs take x_hi·Π_hi + x_hi·Π_lo + x_lo·Π_hi (the dropped
// x_lo·Π_lo is ~2⁻¹⁸ of y); two epilogue warpgroups instead of three.
template <int D, bool F32 = false>
struct TcCfg {
    static constexpr int kChunks = D / kKC;
    static constexpr int kTileBytes = kTile * D * 2;          // one bf16 tile
    static constexpr int kStageBytes = (F32 ? 2 : 1) * kTileBytes;
    static constexpr int kChunkBytesA = kTile * 128;  // one 64-column chunk of a tile
    static constexpr int kChunkBytesB = D * 128;      // one 64-column chunk of Π
    static constexpr int kPiBytes = D * D * 2;
    static constexpr int kStages = F32 ? (D == 64 ? 4 : 2) : (D == 64 ? 8 : 4);
    static constexpr int kAcc = F32 ? 2 : 3;           // TMEM accumulators = epilogue warpgroups
    static constexpr int kConvWarp0 = 2 + 4 * kAcc;    // first converter warp (F32)
    static_assert(32 * (kConvWarp0 + (F32 ? 4 : 0)) == kThreads, "warp roles");
    // allocation: the power of two ≥ kAcc·D columns (≤ 512)
    static constexpr uint32_t kTmemCols = kAcc * D <= 32 ? 32 : (kAcc * D <= 64 ? 64 : (kAcc * D <= 128 ? 128 : (kAcc * D <= 256 ? 256 : 512)));
    static constexpr size_t kBarOffset = 2 * (size_t)kPiBytes + (size_t)kStages * kStageBytes;
    static constexpr size_t kSmemBytes = kBarOffset + 256 + 1024;  // barriers + alignment slack
};

// One quantizer's share of an mse launch: its rows (a tensor map for bf16 rows,
// a pointer for fp32 rows), its rotation operands, codebook and output planes.
struct TcSide {
    CUtensorMap tm_x, tm_pi_hi, tm_pi_lo;
    const float* xf;
    int64_t xf_stride;
    int64_t n_rows;
    float norm_scale;
    Codebook cb;
    uint8_t* codes;
    float* norm_out;
    int* status;
};

// CTAs [0, split) quantize side a, CTAs [split, gridDim.x) side b (the K and V
// rows of one decode step in one launch; a single quantizer passes split =
// gridDim.x).  Both sides share D, b, the row dtype and the number of Π passes.
template <int D, int BM, bool F32 = false>
__global__ void __launch_bounds__(kThreads, 1)
quantize_mse_tc_kernel(const __grid_constant__ TcSide side_a, const __grid_constant__ TcSide side_b, int split,
                       int npass) {
    using C = TcCfg<D, F32>;
    constexpr int kAcc = C::kAcc;
    const bool on_b = (int)blockIdx.x >= split;
    const TcSide& sd = on_b ? side_b : side_a;
    const int cta = on_b ? (int)blockIdx.x - split : (int)blockIdx.x;
    const int ncta = on_b ? (int)gridDim.x - split : split;
    const CUtensorMap* tm_x = &sd.tm_x;
    const CUtensorMap* tm_pi_hi = &sd.tm_pi_hi;
    const CUtensorMap* tm_pi_lo = &sd.tm_pi_lo;
    const int64_t n_rows = sd.n_rows;
    int* const status = sd.status;
    constexpr int L = 1 << BM;
    constexpr int P = L / 2 - 1;          // positive decision boundaries
    constexpr int WORDS = BM * D / 32;    // packed 32-bit words per row
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    allow_dependents();
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* pi_hi = smem;
    uint8_t* pi_lo = smem + C::kPiBytes;
    uint8_t* stages = smem + 2 * C::kPiBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    uint64_t* full = bars;                      // [kStages]
    uint64_t* empty = bars + C::kStages;        // [kStages]
    uint64_t* tfull = empty + C::kStages;       // [kAcc]
    uint64_t* tempty = tfull + kAcc;            // [kAcc]
    uint64_t* pi_full = tempty + kAcc;
    uint64_t* drain = pi_full + 1;  // barrier region: 2·kStages + 2·kAcc + 2 ≤ 26 words
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = (n_rows + kTile - 1) / kTile;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], F32 ? 128 : 1);  // the converter threads, or the TMA's expect_tx
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(pi_full, 1);
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_holder, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ producer
        if (!F32) prefetch_tensormap(tm_x);
        prefetch_tensormap(tm_pi_hi);
        prefetch_tensormap(tm_pi_lo);
        mbar_arrive_expect_tx(pi_full, npass * C::kPiBytes);
        for (int c = 0; c < C::kChunks; ++c) {
            tma_load_2d(pi_hi + c * C::kChunkBytesB, tm_pi_hi, pi_full, c * kKC, 0);
            if (npass == 2) tma_load_2d(pi_lo + c * C::kChunkBytesB, tm_pi_lo, pi_full, c * kKC, 0);
        }
        int64_t i = 0;
        for (int64_t tile = cta; !F32 && tile < ntiles; tile += ncta, ++i) {
            const int s = (int)(i % C::kStages);
            const int64_t u = i / C::kStages;
            if (u > 0 && !mbar_wait(&empty[s], (uint32_t)((u - 1) & 1), status, 1)) break;
            mbar_arrive_expect_tx(&full[s], C::kStageBytes);
            uint8_t* st = stages + (size_t)s * C::kStageBytes;
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_2d(st + c * C::kChunkBytesA, tm_x, &full[s], c * kKC, (int)(tile * kTile));
        }
        // Every load issued must have landed before the CTA may exit.
        const int64_t issued = i;
        for (int64_t k = (issued > C::kStages ? issued - C::kStages : 0); k < issued; ++k)
            mbar_wait(&full[k % C::kStages], (uint32_t)((k / C::kStages) & 1), status, 2);
        mbar_wait(pi_full, 0, status, 2);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(kTile, D);
        bool ok = mbar_wait(pi_full, 0, status, 3);
        tc_fence_after();
        const uint32_t a_base = smem_u32(stages), hi_base = smem_u32(pi_hi), lo_base = smem_u32(pi_lo);
        int64_t i = 0;
        for (int64_t tile = cta; ok && tile < ntiles; tile += ncta, ++i) {
            const int s = (int)(i % C::kStages);
            const int acc = (int)(i % kAcc);
            const int64_t ua = i / kAcc;
            if (!(ok = mbar_wait(&full[s], (uint32_t)((i / C::kStages) & 1), status, 4))) break;
            if (ua > 0 && !(ok = mbar_wait(&tempty[acc], (uint32_t)((ua - 1) & 1), status, 5))) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * D);
            const uint32_t a_stage = a_base + (uint32_t)(s * C::kStageBytes);
            // passes (A, B): bf16 rows (x, Π_hi), (x, Π_lo); fp32 rows also (x_lo, Π_hi);
            // the exact ±1 Walsh–Hadamard operand needs no Π_lo pass
#pragma unroll
            for (int pass = 0; pass < (F32 ? 3 : 2); ++pass) {
                const bool pi_lo_pass = pass == 1;
                if (pi_lo_pass && npass < 2) continue;
                const uint32_t b_base = pi_lo_pass ? lo_base : hi_base;
                const uint32_t a_tile = a_stage + (pass == 2 ? (uint32_t)C::kTileBytes : 0u);
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c)
#pragma unroll
                    for (int kk = 0; kk < kKC / 16; ++kk) {
                        const uint64_t ad = smem_desc(a_tile + c * C::kChunkBytesA + kk * 32, 1024, 2);
                        const uint64_t bd = smem_desc(b_base + c * C::kChunkBytesB + kk * 32, 1024, 2);
                        mma_f16_ss(d_tmem, ad, bd, idesc, (pass | c | kk) != 0);
                    }
            }
            mma_commit(&empty[s]);
            mma_commit(&tfull[acc]);
        }
        mma_commit(drain);
        mbar_wait(drain, 0, status, 6);
    } else if (F32 && warp >= C::kConvWarp0) {
        // ------------------------------------------------------------ converters (fp32 rows)
        // thread ct takes 16-byte chunks (8 columns) ct, ct + 128, … of the tile; each
        // becomes 8 bf16 hi and 8 bf16 lo values at the chunk's 128-byte-swizzled
        // place (row r: 16-byte slot (c8 mod 8) XOR (r mod 8) of its 64-column block)
        const int ct = threadIdx.x - 32 * C::kConvWarp0;
        const float* __restrict__ xf = sd.xf;
        const int64_t xf_stride = sd.xf_stride;
        constexpr int CH = D / 8;  // chunks per row
        constexpr int kRounds = kTile * CH / (128 * 4);
        auto conv_all = [&](bool ok) -> bool {
            uint32_t r;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\t"
                "setp.ne.u32 p, %1, 0;\n\t"
                "bar.red.and.pred q, 1, 128, p;\n\t"
                "selp.u32 %0, 1, 0, q;\n\t}\n"
                : "=r"(r)
                : "r"((uint32_t)ok)
                : "memory");
            return r != 0;
        };
        int64_t i = 0;
        for (int64_t tile = cta; tile < ntiles; tile += ncta, ++i) {
            const int s = (int)(i % C::kStages);
            const int64_t u = i / C::kStages;
            if (u > 0 && !conv_all(mbar_wait(&empty[s], (uint32_t)((u - 1) & 1), status, 8))) break;
            uint8_t* st = stages + (size_t)s * C::kStageBytes;
#pragma unroll
            for (int rd = 0; rd < kRounds; ++rd) {
                float4 v[4][2];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int q = ct + 128 * (4 * rd + k), r = q / CH, c8 = q % CH;
                    const int64_t row = tile * kTile + r;
                    if (row < n_rows) {
                        const float4* src = reinterpret_cast<const float4*>(xf + row * xf_stride + 8 * c8);
                        v[k][0] = __ldg(src);
                        v[k][1] = __ldg(src + 1);
                    } else {
                        v[k][0] = v[k][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int q = ct + 128 * (4 * rd + k), r = q / CH, c8 = q % CH;
                    const float xv[8] = {v[k][0].x, v[k][0].y, v[k][0].z, v[k][0].w,
                                         v[k][1].x, v[k][1].y, v[k][1].z, v[k][1].w};
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(xv[2 * e], xv[2 * e + 1]);
                        const float2 hf = __bfloat1622float2(h2);
                        const __nv_bfloat162 l2 = __floats2bfloat162_rn(xv[2 * e] - hf.x, xv[2 * e + 1] - hf.y);
                        hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
                        lo[e] = *reinterpret_cast<const uint32_t*>(&l2);
                    }
                    uint8_t* dst = st + (c8 / 8) * C::kChunkBytesA + r * 128 + (((c8 % 8) ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4*>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(dst + C::kTileBytes) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
            fence_proxy_async_smem();  // the generic-proxy writes above, before the MMA reads them
            mbar_arrive(&full[s]);
        }
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue
        constexpr int GB = BM == 3 ? 24 : 16;  // bits per float packing group
        constexpr int GC = GB / BM;            // codes per group
        constexpr int NG = 32 / GC;            // groups per 32-code TMEM chunk
        constexpr float kAcc0 = (float)(1u << (GB - 1)) - 0.5f;  // Σ_i (L/2 − ½)·2^(b·i)
        const int wg = (warp - 2) >> 2;                 // accumulator served
        const int quad = warp & 3;                      // TMEM lane quadrant of this warp
        const Codebook& cb = sd.cb;
        uint8_t* const codes = sd.codes;
        float* const norm_out = sd.norm_out;
        const float norm_scale = sd.norm_scale;
        const int r_local = quad * 32 + lane;
        float t2[P > 0 ? P : 1];                        // squared positive boundaries
#pragma unroll
        for (int p = 0; p < P; ++p) t2[p] = cb.t[L / 2 + p] * cb.t[L / 2 + p];
        const uint32_t taddr0 = tmem_base + (uint32_t)(wg * D) + ((uint32_t)(quad * 32) << 16);
        int64_t j = 0;
        for (int64_t tile = cta + (int64_t)wg * ncta; tile < ntiles; tile += (int64_t)kAcc * ncta, ++j) {
            if (!mbar_wait(&tfull[wg], (uint32_t)(j & 1), status, 7)) break;
            tc_fence_after();
            // pass 1: ‖y‖², two 32-column TMEM loads in flight per wait
            uint32_t r[2][32];
            uint64_t ss2 = 0ull;
#pragma unroll
            for (int c = 0; c < D / 32; c += 2) {
                tmem_ld32(taddr0 + c * 32, r[0]);
                tmem_ld32(taddr0 + (c + 1) * 32, r[1]);
                tmem_wait_ld(r[0]);
                tmem_wait_ld(r[1]);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int k = 0; k < 32; k += 2) {
                        const uint64_t v2 = f2(__uint_as_float(r[h][k]), __uint_as_float(r[h][k + 1]));
                        ss2 = fma2(v2, v2, ss2);
                    }
            }
            float ssa, ssb;
            f2_split(ss2, ssa, ssb);
            const float ss = ssa + ssb;
            const float n = sqrtf(ss);
            // c = K/‖y‖² with K = 2^62, lowered for rows so small that c would overflow
            const float cs = ss >= 0x1p-38f ? __fdividef(0x1p62f, ss) : 0x1p100f;
            const float kr = cs * ss;
            const uint64_t cs2 = f2(cs, cs);
            float kt2[P > 0 ? P : 1];
#pragma unroll
            for (int p = 0; p < P; ++p) kt2[p] = -kr * t2[p];
            const int64_t row = tile * kTile + r_local;
            const bool live = row < n_rows;
            // a zero row stores codes 0 (the sign test would give L/2)
            const uint32_t keep = n == 0.f ? 0u : 0xffffffffu;
            uint8_t* dst = codes + row * (int64_t)(WORDS * 4);
            // pass 2: chunk c + 1 is loaded while chunk c is bucketized
            tmem_ld32(taddr0, r[0]);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                tmem_wait_ld(r[c & 1]);
                if (c + 1 < D / 32) tmem_ld32(taddr0 + (c + 1) * 32, r[(c + 1) & 1]);
                const uint32_t* rc = r[c & 1];
                // codes of coordinate pairs (k, k+1); each group keeps an even and an
                // odd partial sum (both exact integers) in one packed accumulator
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
                    acc[k / GC] = fma2(f2(sa, sb),
                                       f2((float)(1u << (BM * (k % GC))), (float)(1u << (BM * ((k + 1) % GC)))),
                                       acc[k / GC]);
                }
                // the chunk's 32 codes are BM consecutive words of the row: store them now
                uint32_t cw[BM];
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
                if (live) {
                    uint8_t* cd = dst + c * (BM * 4);
                    if constexpr (BM == 4) {
                        *reinterpret_cast<uint4*>(cd) = make_uint4(cw[0] & keep, cw[1] & keep, cw[2] & keep, cw[3] & keep);
                    } else if constexpr (BM == 2) {
                        *reinterpret_cast<uint2*>(cd) = make_uint2(cw[0] & keep, cw[1] & keep);
                    } else {
#pragma unroll
                        for (int w = 0; w < BM; ++w) reinterpret_cast<uint32_t*>(cd)[w] = cw[w] & keep;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[wg]);
            if (live) norm_out[row] = n * norm_scale;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

TcSide make_side(const tq_ctx& h, const CUtensorMap* tm_x, const float* xf, int64_t stride, int64_t n_rows,
                 const tq_planes& out) {
    TcSide sd;
    memset(&sd, 0, sizeof(sd));
    const bool one = h.rot_passes == 1;
    if (tm_x) sd.tm_x = *tm_x;
    sd.tm_pi_hi = one ? h.dp.tm_pm : h.dp.tm_pi_hi;
    sd.tm_pi_lo = one ? h.dp.tm_pm : h.dp.tm_pi_lo;
    sd.xf = xf;
    sd.xf_stride = stride;
    sd.n_rows = n_rows;
    sd.norm_scale = h.rot_norm_scale;
    sd.cb = h.cb;
    sd.codes = out.codes;
    sd.norm_out = out.norm;
    sd.status = h.dp.status;
    return sd;
}

// One launch over one side, or over two (b != nullptr, both holding rows): the
// grid's CTAs are divided between the sides in proportion to their tiles.
template <int D, int BM, bool F32>
int launch_tc(const TcSide& a, const TcSide* b, int npass, int num_sms, cudaStream_t s) {
    using C = TcCfg<D, F32>;
    auto fn = quantize_mse_tc_kernel<D, BM, F32>;
    static std::atomic<uint64_t> smem_set{0};
    const int rc = ensure_smem_attr(smem_set, (const void*)fn, (int)C::kSmemBytes, "quantize smem attribute");
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
    fn<<<grid, kThreads, C::kSmemBytes, s>>>(a, b ? *b : a, split, npass);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "tensor-core quantize launch");
}

template <int D, int BM>
int launch_tc(const tq_ctx& h, const CUtensorMap& tm_x, int64_t n_rows, const tq_planes& out, cudaStream_t s) {
    const TcSide a = make_side(h, &tm_x, nullptr, 0, n_rows, out);
    return launch_tc<D, BM, false>(a, nullptr, h.rot_passes, h.num_sms, s);
}

template <int D>
int launch_tc_d(const tq_ctx& h, const CUtensorMap& tm_x, int64_t n_rows, const tq_planes& out, cudaStream_t s) {
    switch (h.hp.b_mse) {
        case 1: return launch_tc<D, 1>(h, tm_x, n_rows, out, s);
        case 2: return launch_tc<D, 2>(h, tm_x, n_rows, out, s);
        case 3: return launch_tc<D, 3>(h, tm_x, n_rows, out, s);
        case 4: return launch_tc<D, 4>(h, tm_x, n_rows, out, s);
        default: return fail(TQ_EUNSUPPORTED, "b_m=%d", h.hp.b_mse);
    }
}

// fp32 rows (mse, d = 64 and 128): the rows are read by the kernel's converter
// warps; the X tensor map is unused
template <int D>
int launch_tc_f32_d(const tq_ctx& h, const float* x, int64_t n_rows, int64_t stride, const tq_planes& out,
                    cudaStream_t s) {
    const TcSide a = make_side(h, nullptr, x, stride, n_rows, out);
    switch (h.hp.b_mse) {
        case 1: return launch_tc<D, 1, true>(a, nullptr, h.rot_passes, h.num_sms, s);
        case 2: return launch_tc<D, 2, true>(a, nullptr, h.rot_passes, h.num_sms, s);
        case 3: return launch_tc<D, 3, true>(a, nullptr, h.rot_passes, h.num_sms, s);
        case 4: return launch_tc<D, 4, true>(a, nullptr, h.rot_passes, h.num_sms, s);
        default: return fail(TQ_EUNSUPPORTED, "b_m=%d", h.hp.b_mse);
    }
}

// K and V sides in one launch (same D, b, row dtype and Π passes)
template <int D, bool F32>
int launch_tc_pair_d(int b_mse, const TcSide& a, const TcSide& b, int npass, int num_sms, cudaStream_t s) {
    switch (b_mse) {
        case 1: return launch_tc<D, 1, F32>(a, &b, npass, num_sms, s);
        case 2: return launch_tc<D, 2, F32>(a, &b, npass, num_sms, s);
        case 3: return launch_tc<D, 3, F32>(a, &b, npass, num_sms, s);
        case 4: return launch_tc<D, 4, F32>(a, &b, npass, num_sms, s);
        default: return fail(TQ_EUNSUPPORTED, "b_m=%d", b_mse);
    }
}


// ---------------------------------------------------------------------------
// d = 256, mse: Π_hi + Π_lo (256 KB of bf16) do not fit beside the row tiles, so
// Π is streamed with them.  A stage holds 64-dim chunk c of a 128-row tile and
// the same 64 columns of Π_hi and Π_lo (all 256 output rows, 128-byte swizzled);
// per k16 step and pass one N = 256 MMA accumulates Y = X·Πᵀ over the four chunks
// into one of two 256-column TMEM slots.  Four epilogue warpgroups, two per slot,
// each take half of the columns; the halves of ‖y‖² meet in shared memory behind
// a named barrier.  Π is re-read from L2 for every tile: 256 KB per 128 rows,
// which keeps this path near the tensor and L2 rates rather than HBM's.
constexpr int k256Stages = 2;
constexpr int k256EpiWarps = 16;
constexpr int k256Threads = 32 * (2 + k256EpiWarps);

struct Cfg256 {
    static constexpr int D = 256;
    static constexpr int kChunks = D / kKC;                      // 4
    static constexpr int kXBytes = kTile * 128;                  // 16 KB: 128 rows × 64 bf16
    static constexpr int kPBytes = D * 128;                      // 32 KB: 256 rows × 64 bf16
    static constexpr int kStageBytes = kXBytes + 2 * kPBytes;    // 80 KB
    static constexpr size_t kBarOffset = (size_t)k256Stages * kStageBytes;
    static constexpr size_t kXchOffset = kBarOffset + 256;      // [slot][half][row] partial ‖y‖²
    static constexpr size_t kSmemBytes = kXchOffset + (size_t)2 * 2 * kTile * 4 + 1024;
};

template <int BM>
__global__ void __launch_bounds__(k256Threads, 1)
quantize_mse_tc256_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_pi_hi,
                          const __grid_constant__ CUtensorMap tm_pi_lo, int64_t n_rows, int npass, float norm_scale,
                          Codebook cb, uint8_t* __restrict__ codes, float* __restrict__ norm_out,
                          int* __restrict__ status) {
    using C = Cfg256;
    constexpr int D = C::D;
    constexpr int H = D / 2;              // columns per half
    constexpr int L = 1 << BM;
    constexpr int P = L / 2 - 1;          // positive decision boundaries
    constexpr int WORDS = BM * D / 32;    // packed 32-bit words per row
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    allow_dependents();
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    uint64_t* full = bars;                 // [k256Stages] chunk landed
    uint64_t* empty = full + k256Stages;   // [k256Stages] chunk consumed by the MMAs
    uint64_t* tfull = empty + k256Stages;  // [2] Y ready
    uint64_t* tempty = tfull + 2;          // [2] slot read out (256 arrivals)
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = (n_rows + kTile - 1) / kTile;

    if (threadIdx.x == 0) {
        for (int s = 0; s < k256Stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 256);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ producer
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_pi_hi);
        prefetch_tensormap(&tm_pi_lo);
        int64_t q = 0;  // chunks issued
        bool ok = true;
        for (int64_t tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
            for (int c = 0; c < C::kChunks; ++c, ++q) {
                const int s = (int)(q % k256Stages);
                const int64_t u = q / k256Stages;
                if (u > 0 && !(ok = mbar_wait(&empty[s], (uint32_t)((u - 1) & 1), status, 21))) break;
                uint8_t* st = stages + (size_t)s * C::kStageBytes;
                mbar_arrive_expect_tx(&full[s], C::kXBytes + npass * C::kPBytes);
                tma_load_2d(st, &tm_x, &full[s], c * kKC, (int)(tile * kTile));
                tma_load_2d(st + C::kXBytes, &tm_pi_hi, &full[s], c * kKC, 0);
                if (npass == 2) tma_load_2d(st + C::kXBytes + C::kPBytes, &tm_pi_lo, &full[s], c * kKC, 0);
            }
        }
        // every load issued must have landed before the CTA may exit
        for (int64_t k = (q > k256Stages ? q - k256Stages : 0); k < q; ++k)
            mbar_wait(&full[k % k256Stages], (uint32_t)((k / k256Stages) & 1), status, 22);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(kTile, D);
        const uint32_t base = smem_u32(stages);
        int64_t q = 0, i = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++i) {
            const int a = (int)(i & 1);
            const int64_t ua = i >> 1;
            if (ua > 0 && !(ok = mbar_wait(&tempty[a], (uint32_t)((ua - 1) & 1), status, 23))) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(a * D);
            for (int c = 0; c < C::kChunks; ++c, ++q) {
                const int s = (int)(q % k256Stages);
                if (!(ok = mbar_wait(&full[s], (uint32_t)((q / k256Stages) & 1), status, 24))) break;
                tc_fence_after();
                const uint32_t st = base + (uint32_t)(s * C::kStageBytes);
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    if (pass >= npass) break;
#pragma unroll
                    for (int kk = 0; kk < kKC / 16; ++kk) {
                        const uint64_t ad = smem_desc(st + kk * 32, 1024, 2);
                        const uint64_t bd = smem_desc(st + C::kXBytes + pass * C::kPBytes + kk * 32, 1024, 2);
                        mma_f16_ss(d_tmem, ad, bd, idesc, (c | kk | pass) != 0);
                    }
                }
                mma_commit(&empty[s]);
            }
            if (ok) mma_commit(&tfull[a]);
        }
        mma_commit(drain);
        mbar_wait(drain, 0, status, 25);
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue
        constexpr int GB = BM == 3 ? 24 : 16;  // bits per float packing group
        constexpr int GC = GB / BM;            // codes per group
        constexpr int NG = 32 / GC;            // groups per 32-code TMEM chunk
        constexpr float kAcc0 = (float)(1u << (GB - 1)) - 0.5f;
        const int wg = (warp - 2) >> 2;        // 0..3
        const int slot = wg >> 1, half = wg & 1;
        const int quad = warp & 3;             // TMEM lane quadrant of this warp
        const int r_local = quad * 32 + lane;
        float* xss = reinterpret_cast<float*>(smem + C::kXchOffset) + slot * (2 * kTile);  // [half][row]
        float t2[P > 0 ? P : 1];
#pragma unroll
        for (int p = 0; p < P; ++p) t2[p] = cb.t[L / 2 + p] * cb.t[L / 2 + p];
        const uint32_t ybase = tmem_base + (uint32_t)(slot * D + half * H) + ((uint32_t)(quad * 32) << 16);
        auto pair_sync = [&]() { asm volatile("bar.sync %0, 256;" ::"r"(1 + slot) : "memory"); };
        // the two halves of a slot leave the tile loop together when a wait gives up
        auto pair_all = [&](bool ok) -> bool {
            uint32_t r;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\t"
                "setp.ne.u32 p, %1, 0;\n\t"
                "bar.red.and.pred q, %2, 256, p;\n\t"
                "selp.u32 %0, 1, 0, q;\n\t}\n"
                : "=r"(r)
                : "r"((uint32_t)ok), "r"(1 + slot)
                : "memory");
            return r != 0;
        };
        int64_t j = 0;
        for (int64_t tile = blockIdx.x + (int64_t)slot * gridDim.x; tile < ntiles; tile += 2 * (int64_t)gridDim.x, ++j) {
            if (!pair_all(mbar_wait(&tfull[slot], (uint32_t)(j & 1), status, 26))) break;
            tc_fence_after();
            uint32_t r[2][32];
            // pass 1: this half's part of ‖y‖², summed with the other half's
            uint64_t ss2 = 0ull;
#pragma unroll
            for (int c = 0; c < H / 32; c += 2) {
                tmem_ld32(ybase + c * 32, r[0]);
                tmem_ld32(ybase + (c + 1) * 32, r[1]);
                tmem_wait_ld(r[0]);
                tmem_wait_ld(r[1]);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int k = 0; k < 32; k += 2) {
                        const uint64_t v2 = f2(__uint_as_float(r[h][k]), __uint_as_float(r[h][k + 1]));
                        ss2 = fma2(v2, v2, ss2);
                    }
            }
            float ssa, ssb;
            f2_split(ss2, ssa, ssb);
            xss[half * kTile + r_local] = ssa + ssb;
            pair_sync();
            const float ss = xss[r_local] + xss[kTile + r_local];  // same order in both halves
            const float n = sqrtf(ss);
            const float cs = ss >= 0x1p-38f ? __fdividef(0x1p62f, ss) : 0x1p100f;
            const float kr = cs * ss;
            const uint64_t cs2 = f2(cs, cs);
            float kt2[P > 0 ? P : 1];
#pragma unroll
            for (int p = 0; p < P; ++p) kt2[p] = -kr * t2[p];
            const int64_t row = tile * kTile + r_local;
            const bool live = row < n_rows;
            const uint32_t keep = n == 0.f ? 0u : 0xffffffffu;
            uint8_t* dst = codes + row * (int64_t)(WORDS * 4) + half * (H / 32) * (BM * 4);
            // pass 2: chunk c + 1 is loaded while chunk c is bucketized
            tmem_ld32(ybase, r[0]);
#pragma unroll
            for (int c = 0; c < H / 32; ++c) {
                tmem_wait_ld(r[c & 1]);
                if (c + 1 < H / 32) tmem_ld32(ybase + (c + 1) * 32, r[(c + 1) & 1]);
                const uint32_t* rc = r[c & 1];
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
                    float ca, cb2;
                    f2_split(cnt2, ca, cb2);
                    const float sa = __uint_as_float(__float_as_uint(ca) | (__float_as_uint(va) & 0x80000000u));
                    const float sb = __uint_as_float(__float_as_uint(cb2) | (__float_as_uint(vb) & 0x80000000u));
                    acc[k / GC] = fma2(f2(sa, sb),
                                       f2((float)(1u << (BM * (k % GC))), (float)(1u << (BM * ((k + 1) % GC)))),
                                       acc[k / GC]);
                }
                uint32_t cw[BM];
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
                if (live) {
                    uint8_t* cd = dst + c * (BM * 4);
                    if constexpr (BM == 4) {
                        *reinterpret_cast<uint4*>(cd) = make_uint4(cw[0] & keep, cw[1] & keep, cw[2] & keep, cw[3] & keep);
                    } else if constexpr (BM == 2) {
                        *reinterpret_cast<uint2*>(cd) = make_uint2(cw[0] & keep, cw[1] & keep);
                    } else {
#pragma unroll
                        for (int w = 0; w < BM; ++w) reinterpret_cast<uint32_t*>(cd)[w] = cw[w] & keep;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[slot]);
            if (live && half == 0) norm_out[row] = n * norm_scale;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

template <int BM>
int launch_tc256(const tq_ctx& h, const CUtensorMap& tm_x, int64_t n_rows, const tq_planes& out, cudaStream_t s) {
    using C = Cfg256;
    static_assert(C::kSmemBytes <= 232448, "d = 256 quantize shared memory above the per-CTA limit");
    auto fn = quantize_mse_tc256_kernel<BM>;
    static std::atomic<uint64_t> smem_set{0};
    const int rc = ensure_smem_attr(smem_set, (const void*)fn, (int)C::kSmemBytes, "d=256 quantize smem attribute");
    if (rc != TQ_OK) return rc;
    const int64_t ntiles = (n_rows + kTile - 1) / kTile;
    const int grid = (int)(ntiles < h.num_sms ? ntiles : h.num_sms);
    const bool one = h.rot_passes == 1;
    fn<<<grid, k256Threads, C::kSmemBytes, s>>>(tm_x, one ? h.dp.tm_pm : h.dp.tm_pi_hi, one ? h.dp.tm_pm : h.dp.tm_pi_lo,
                                                n_rows, h.rot_passes, h.rot_norm_scale, h.cb, out.codes, out.norm,
                                                h.dp.status);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "d=256 tensor-core quantize launch");
}

int launch_tc256_b(const tq_ctx& h, const CUtensorMap& tm_x, int64_t n_rows, const tq_planes& out, cudaStream_t s) {
    switch (h.hp.b_mse) {
        case 1: return launch_tc256<1>(h, tm_x, n_rows, out, s);
        case 2: return launch_tc256<2>(h, tm_x, n_rows, out, s);
        case 3: return launch_tc256<3>(h, tm_x, n_rows, out, s);
        case 4: return launch_tc256<4>(h, tm_x, n_rows, out, s);
        default: return fail(TQ_EUNSUPPORTED, "b_m=%d", h.hp.b_mse);
    }
}

// ---------------------------------------------------------------------------
// The prod variant («Собственно TurboQuant»): codes with b_m = b − 1 bits as
// above, plus the QJL sketch of the rotated unit residual e = y/‖y‖ − c[idx]:
// signs = [T·e ≥ 0] with T = S·Πᵀ, and ‖r‖ = ‖e‖ (Π orthogonal).
//
// Per 128-row tile and TMEM slot (2·D columns: Y, later E, then S):
//   MMA 1  Y = X·Πᵀ (bf16 hi/lo of Π, as above)              → columns [0, D)
//   epilogue pass 1/2: ‖y‖, codes, and e = y/‖y‖ − c[idx] written back as f16
//          hi/lo pairs into the Y columns already read (32-dim chunk k: hi in
//          columns 32k … 32k + 15, lo in 32k + 16 … 32k + 31)
//   MMA 2  S = E·Tᵀ with A read from tensor memory, three f16 passes
//          E_hi·T_hi + E_lo·T_hi + E_hi·T_lo (≈2⁻²² relative)   → columns [D, 2D)
//   epilogue pass 3: sign bits of S.
// Warps: 0 TMA producer (Π, T once, then X tiles), 1 TMEM owner and MMA issuer,
// 2..17 four epilogue warpgroups: two per TMEM slot, each taking half of the
// columns of the slot's 128 rows (the row norms are summed through shared memory).
constexpr int kProdSlots = 2;
constexpr int kProdEpiWarps = 8 * kProdSlots;
constexpr int kProdThreads = 32 * (2 + kProdEpiWarps);

template <int D>
struct ProdCfg {
    static constexpr int kChunks = D / kKC;
    static constexpr int kStageBytes = kTile * D * 2;
    static constexpr int kChunkBytesA = kTile * 128;
    static constexpr int kChunkBytesB = D * 128;
    static constexpr int kMatBytes = D * D * 2;
    static constexpr int kStages = D == 64 ? 4 : 2;
    static constexpr uint32_t kTmemCols = kProdSlots * 2 * D;  // 256 or 512
    static constexpr size_t kBarOffset = 4 * (size_t)kMatBytes + (size_t)kStages * kStageBytes;
    static constexpr size_t kXchOffset = kBarOffset + 256;  // [slot][2 sums][2 halves][128 rows] floats
    static constexpr size_t kSmemBytes = kXchOffset + (size_t)kProdSlots * 2 * 2 * kTile * 4 + 1024;
};

// The positive centroids c⁺_k (k = 0 … L/2 − 1) as a polynomial in the bucket
// counter value x = k + ½ (what the saturated boundary tests sum to), interpolating
// the L/2 points and built in double precision, so that a residual takes one packed
// Horner step per degree.  Coefficients are stored negated and per row multiplied
// by 0 for a zero row, whose residual must be 0.
template <int BM>
struct CentroidPoly {
    static constexpr int N = BM >= 1 ? (1 << (BM - 1)) : 1;
    float m[N];  // −(monomial coefficients), m[0] constant term
    __device__ void init(const Codebook& cb) {
        constexpr int L = 1 << BM;
        double v[N], P[N];
#pragma unroll
        for (int k = 0; k < N; ++k) v[k] = BM >= 1 ? (double)cb.c[L / 2 + k] : 0.0;
        // Newton divided differences on the nodes k + ½ (unit spacing)
#pragma unroll
        for (int j = 1; j < N; ++j)
#pragma unroll
            for (int k = N - 1; k >= j; --k) v[k] = (v[k] - v[k - 1]) / (double)j;
        // expand p(x) = v0 + v1 (x − x0) + v2 (x − x0)(x − x1) + … into monomials
#pragma unroll
        for (int k = 0; k < N; ++k) P[k] = 0.0;
        P[0] = v[N - 1];
#pragma unroll
        for (int j = N - 2; j >= 0; --j) {
            const double xj = j + 0.5;
#pragma unroll
            for (int i = N - 1; i >= 1; --i) P[i] = P[i - 1] - xj * P[i];
            P[0] = v[j] - xj * P[0];
        }
#pragma unroll
        for (int k = 0; k < N; ++k) m[k] = (float)-P[k];
    }
};

template <int D, int BM>
__global__ void __launch_bounds__(kProdThreads, 1)
quantize_prod_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_pi_hi,
                        const __grid_constant__ CUtensorMap tm_pi_lo, const __grid_constant__ CUtensorMap tm_t_hi,
                        const __grid_constant__ CUtensorMap tm_t_lo, int64_t n_rows, int npass, float norm_scale,
                        Codebook cb,
                        uint8_t* __restrict__ codes, uint8_t* __restrict__ signs, float* __restrict__ norm_out,
                        float* __restrict__ rnorm_out, int* __restrict__ status) {
    using C = ProdCfg<D>;
    constexpr int L = 1 << BM;
    constexpr int P = BM >= 1 ? L / 2 - 1 : 0;  // positive decision boundaries
    constexpr int WORDS = BM * D / 32;          // packed code words per row
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    allow_dependents();
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* pi_hi = smem;
    uint8_t* pi_lo = smem + C::kMatBytes;
    uint8_t* t_hi = smem + 2 * C::kMatBytes;
    uint8_t* t_lo = smem + 3 * C::kMatBytes;
    uint8_t* stages = smem + 4 * C::kMatBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    uint64_t* full = bars;                        // [kStages] X tile landed
    uint64_t* empty = full + C::kStages;          // [kStages] X tile consumed by MMA 1
    uint64_t* yfull = empty + C::kStages;         // [slots] Y ready
    uint64_t* efull = yfull + kProdSlots;         // [slots] E written (128 arrivals)
    uint64_t* sfull = efull + kProdSlots;         // [slots] S ready
    uint64_t* sfree = sfull + kProdSlots;         // [slots] slot read out (128 arrivals)
    uint64_t* mat_full = sfree + kProdSlots;
    uint64_t* drain = mat_full + 1;               // ≤ 2·6 + 8 + 2 = 22 words
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = (n_rows + kTile - 1) / kTile;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < kProdSlots; ++a) {
            mbar_init(&yfull[a], 1);
            mbar_init(&efull[a], 256);
            mbar_init(&sfull[a], 1);
            mbar_init(&sfree[a], 256);
        }
        mbar_init(mat_full, 1);
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_holder, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ producer
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_pi_hi);
        prefetch_tensormap(&tm_pi_lo);
        prefetch_tensormap(&tm_t_hi);
        prefetch_tensormap(&tm_t_lo);
        mbar_arrive_expect_tx(mat_full, (2 + npass) * C::kMatBytes);
        for (int c = 0; c < C::kChunks; ++c) {
            tma_load_2d(pi_hi + c * C::kChunkBytesB, &tm_pi_hi, mat_full, c * kKC, 0);
            if (npass == 2) tma_load_2d(pi_lo + c * C::kChunkBytesB, &tm_pi_lo, mat_full, c * kKC, 0);
            tma_load_2d(t_hi + c * C::kChunkBytesB, &tm_t_hi, mat_full, c * kKC, 0);
            tma_load_2d(t_lo + c * C::kChunkBytesB, &tm_t_lo, mat_full, c * kKC, 0);
        }
        int64_t i = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
            const int s = (int)(i % C::kStages);
            const int64_t u = i / C::kStages;
            if (u > 0 && !mbar_wait(&empty[s], (uint32_t)((u - 1) & 1), status, 11)) break;
            mbar_arrive_expect_tx(&full[s], C::kStageBytes);
            uint8_t* st = stages + (size_t)s * C::kStageBytes;
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_2d(st + c * C::kChunkBytesA, &tm_x, &full[s], c * kKC, (int)(tile * kTile));
        }
        // every load issued must have landed before the CTA may exit
        const int64_t issued = i;
        for (int64_t k = (issued > C::kStages ? issued - C::kStages : 0); k < issued; ++k)
            mbar_wait(&full[k % C::kStages], (uint32_t)((k / C::kStages) & 1), status, 12);
        mbar_wait(mat_full, 0, status, 12);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc1 = idesc_bf16_f32(kTile, D);
        constexpr uint32_t idesc2 = idesc_f16_f32(kTile, D);
        bool ok = mbar_wait(mat_full, 0, status, 13);
        tc_fence_after();
        const uint32_t a_base = smem_u32(stages), pih = smem_u32(pi_hi), pil = smem_u32(pi_lo);
        const uint32_t th = smem_u32(t_hi), tl = smem_u32(t_lo);
        // MMA 2 of tile k: S = E·Tᵀ once the epilogue has written E into the slot
        auto second = [&](int64_t k) {
            const int a = (int)(k % kProdSlots);
            const int64_t ua = k / kProdSlots;
            if (!(ok = mbar_wait(&efull[a], (uint32_t)(ua & 1), status, 14))) return;
            tc_fence_after();
            const uint32_t e_tmem = tmem_base + (uint32_t)(a * 2 * D);
            const uint32_t s_tmem = e_tmem + (uint32_t)D;
#pragma unroll
            for (int pass = 0; pass < 3; ++pass) {
                const uint32_t b_base = pass == 2 ? tl : th;
#pragma unroll
                for (int k16 = 0; k16 < D / 16; ++k16) {
                    // E_hi of dims 16·k16 … in columns 32·(k16/2) + 8·(k16%2), E_lo 16 columns further
                    const uint32_t acol = 32 * (k16 >> 1) + 8 * (k16 & 1) + (pass == 1 ? 16 : 0);
                    const uint64_t bd = smem_desc(b_base + (k16 >> 2) * C::kChunkBytesB + (k16 & 3) * 32, 1024, 2);
                    mma_f16_ts(s_tmem, e_tmem + acol, bd, idesc2, (pass | k16) != 0);
                }
            }
            mma_commit(&sfull[a]);
        };
        int64_t i = 0;
        for (int64_t tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++i) {
            const int s = (int)(i % C::kStages);
            const int a = (int)(i % kProdSlots);
            const int64_t ua = i / kProdSlots;
            if (!(ok = mbar_wait(&full[s], (uint32_t)((i / C::kStages) & 1), status, 15))) break;
            if (ua > 0 && !(ok = mbar_wait(&sfree[a], (uint32_t)((ua - 1) & 1), status, 16))) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(a * 2 * D);
            const uint32_t a_stage = a_base + (uint32_t)(s * C::kStageBytes);
#pragma unroll
            for (int pass = 0; pass < 2; ++pass) {
                if (pass >= npass) break;
                const uint32_t b_base = pass == 0 ? pih : pil;
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c)
#pragma unroll
                    for (int kk = 0; kk < kKC / 16; ++kk) {
                        const uint64_t ad = smem_desc(a_stage + c * C::kChunkBytesA + kk * 32, 1024, 2);
                        const uint64_t bd = smem_desc(b_base + c * C::kChunkBytesB + kk * 32, 1024, 2);
                        mma_f16_ss(d_tmem, ad, bd, idesc1, (pass | c | kk) != 0);
                    }
            }
            mma_commit(&empty[s]);
            mma_commit(&yfull[a]);
            if (i > 0) second(i - 1);
        }
        if (ok && i > 0) second(i - 1);
        mma_commit(drain);
        mbar_wait(drain, 0, status, 17);
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue
        constexpr int GB = BM == 3 ? 24 : 16;  // bits per float packing group
        constexpr int GC = BM > 0 ? GB / BM : 1;
        constexpr int NG = BM > 0 ? 32 / GC : 1;
        constexpr float kAcc0 = (float)(1u << (GB - 1)) - 0.5f;
        constexpr int H = D / 2;                // columns per half
        const int wg = (warp - 2) >> 2;         // 0..3
        const int slot = wg >> 1, half = wg & 1;
        const int quad = warp & 3;              // TMEM lane quadrant of this warp
        const int r_local = quad * 32 + lane;
        float* xch = reinterpret_cast<float*>(smem + C::kXchOffset) + slot * (2 * 2 * kTile);
        float* xss = xch;                       // [half][row] partial ‖y‖²
        float* xes = xch + 2 * kTile;           // [half][row] partial ‖e‖²
        float t2[P > 0 ? P : 1];
#pragma unroll
        for (int p = 0; p < P; ++p) t2[p] = cb.t[L / 2 + p] * cb.t[L / 2 + p];
        CentroidPoly<BM> cp;
        cp.init(cb);
        const uint32_t lanebits = (uint32_t)(quad * 32) << 16;
        const uint32_t ybase = tmem_base + (uint32_t)(slot * 2 * D + half * H) + lanebits;
        const uint32_t sbase = ybase + (uint32_t)D;
        auto pair_sync = [&]() { asm volatile("bar.sync %0, 256;" ::"r"(1 + slot) : "memory"); };
        // Both halves of a slot meet at the named barrier above, so a bounded wait
        // that gives up must end the loop for all 256 threads at once: each wait's
        // outcome is AND-reduced over the pair on the same barrier, and the loop is
        // left only when the reduced result says so.
        auto pair_all = [&](bool ok) -> bool {
            uint32_t r;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\t"
                "setp.ne.u32 p, %1, 0;\n\t"
                "bar.red.and.pred q, %2, 256, p;\n\t"
                "selp.u32 %0, 1, 0, q;\n\t}\n"
                : "=r"(r)
                : "r"((uint32_t)ok), "r"(1 + slot)
                : "memory");
            return r != 0;
        };
        int64_t j = 0;
        for (int64_t tile = blockIdx.x + (int64_t)slot * gridDim.x; tile < ntiles;
             tile += (int64_t)kProdSlots * gridDim.x, ++j) {
            if (!pair_all(mbar_wait(&yfull[slot], (uint32_t)(j & 1), status, 18))) break;
            tc_fence_after();
            uint32_t r[2][32];
            // pass 1: this half's part of ‖y‖², summed with the other half's
            uint64_t ss2 = 0ull;
#pragma unroll
            for (int c = 0; c < H / 32; ++c) tmem_ld32(ybase + c * 32, r[c & 1]);
#pragma unroll
            for (int c = 0; c < H / 32; ++c) {
                tmem_wait_ld(r[c & 1]);
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    const uint64_t v2 = f2(__uint_as_float(r[c & 1][k]), __uint_as_float(r[c & 1][k + 1]));
                    ss2 = fma2(v2, v2, ss2);
                }
            }
            float ssa, ssb;
            f2_split(ss2, ssa, ssb);
            xss[half * kTile + r_local] = ssa + ssb;
            pair_sync();
            const float ss = xss[r_local] + xss[kTile + r_local];  // same order in both halves
            const float n = sqrtf(ss);
            const float inv = n > 0.f ? 1.f / n : 0.f;
            const uint64_t inv2 = f2(inv, inv);
            const float cs = ss >= 0x1p-38f ? __fdividef(0x1p62f, ss) : 0x1p100f;
            const float kr = cs * ss;
            const uint64_t cs2 = f2(cs, cs);
            float kt2[P > 0 ? P : 1];
#pragma unroll
            for (int p = 0; p < P; ++p) kt2[p] = -kr * t2[p];
            const int64_t row = tile * kTile + r_local;
            const bool live = row < n_rows;
            const uint32_t keep = n == 0.f ? 0u : 0xffffffffu;
            // −c⁺ polynomial of this row (all zero for a zero row)
            const float live_f = n > 0.f ? 1.f : 0.f;
            uint64_t nc2[CentroidPoly<BM>::N];
#pragma unroll
            for (int k = 0; k < CentroidPoly<BM>::N; ++k) nc2[k] = f2(cp.m[k] * live_f, cp.m[k] * live_f);
            uint64_t es2 = 0ull;
            // pass 2: chunk c + 1 is loaded while chunk c is bucketized and its residual stored
            tmem_ld32(ybase, r[0]);
#pragma unroll
            for (int c = 0; c < H / 32; ++c) {
                tmem_wait_ld(r[c & 1]);
                if (c + 1 < H / 32) tmem_ld32(ybase + (c + 1) * 32, r[(c + 1) & 1]);
                const uint32_t* rc = r[c & 1];
                uint64_t acc[NG];
#pragma unroll
                for (int gi = 0; gi < NG; ++gi) acc[gi] = f2(kAcc0, 0.f);
                uint32_t ehi[16], elo[16];
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    const float va = __uint_as_float(rc[k]), vb = __uint_as_float(rc[k + 1]);
                    const uint64_t v2 = f2(va, vb);
                    uint64_t cnt2 = f2(0.5f, 0.5f);
                    if constexpr (P > 0) {
                        float wa, wb;
                        f2_split(mul2(v2, cs2), wa, wb);
#pragma unroll
                        for (int p = 0; p < P; ++p)
                            cnt2 = add2(cnt2, f2(__saturatef(fmaf(va, wa, kt2[p])), __saturatef(fmaf(vb, wb, kt2[p]))));
                    }
                    const uint32_t sga = __float_as_uint(va) & 0x80000000u, sgb = __float_as_uint(vb) & 0x80000000u;
                    uint64_t e2;
                    if constexpr (BM > 0) {
                        float ca, cb2;
                        f2_split(cnt2, ca, cb2);
                        const float sa = __uint_as_float(__float_as_uint(ca) | sga);
                        const float sb = __uint_as_float(__float_as_uint(cb2) | sgb);
                        acc[k / GC] = fma2(f2(sa, sb),
                                           f2((float)(1u << (BM * (k % GC))), (float)(1u << (BM * ((k + 1) % GC)))),
                                           acc[k / GC]);
                        // residual e = sign(y)·(|y|/‖y‖ − c⁺(count)) (0 for a zero row)
                        constexpr int N = CentroidPoly<BM>::N;
                        uint64_t nc = nc2[N - 1];
#pragma unroll
                        for (int q = N - 2; q >= 0; --q) nc = fma2(nc, cnt2, nc2[q]);
                        float ta, tb;
                        f2_split(fma2(f2(fabsf(va), fabsf(vb)), inv2, nc), ta, tb);
                        e2 = f2(__uint_as_float(__float_as_uint(ta) ^ sga), __uint_as_float(__float_as_uint(tb) ^ sgb));
                    } else {
                        e2 = mul2(v2, inv2);
                    }
                    es2 = fma2(e2, e2, es2);
                    float ea, eb;
                    f2_split(e2, ea, eb);
                    const __half2 hi = __floats2half2_rn(ea, eb);
                    const float2 hf = __half22float2(hi);
                    const __half2 lo = __floats2half2_rn(ea - hf.x, eb - hf.y);
                    ehi[k / 2] = *reinterpret_cast<const uint32_t*>(&hi);
                    elo[k / 2] = *reinterpret_cast<const uint32_t*>(&lo);
                }
                // the residual of these 32 dims replaces their (already read) Y columns
                tmem_st16(ybase + c * 32, ehi);
                tmem_st16(ybase + c * 32 + 16, elo);
                if constexpr (BM > 0) {
                    uint32_t cw[BM];
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
                    if (live) {
                        uint8_t* cd = codes + row * (int64_t)(WORDS * 4) + (half * (H / 32) + c) * (BM * 4);
                        if constexpr (BM == 2) {
                            *reinterpret_cast<uint2*>(cd) = make_uint2(cw[0] & keep, cw[1] & keep);
                        } else {
#pragma unroll
                            for (int w = 0; w < BM; ++w) reinterpret_cast<uint32_t*>(cd)[w] = cw[w] & keep;
                        }
                    }
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&efull[slot]);
            float esa, esb;
            f2_split(es2, esa, esb);
            xes[half * kTile + r_local] = esa + esb;
            pair_sync();
            if (live && half == 0) {
                norm_out[row] = n * norm_scale;
                rnorm_out[row] = sqrtf(xes[r_local] + xes[kTile + r_local]);
            }
            // pass 3: sign bits of this half of S = T·e (bit i set ⇔ s_i ≥ 0)
            if (!pair_all(mbar_wait(&sfull[slot], (uint32_t)(j & 1), status, 19))) break;
            tc_fence_after();
            uint32_t sw[H / 32];
#pragma unroll
            for (int c = 0; c < H / 32; ++c) tmem_ld32(sbase + c * 32, r[c & 1]);
#pragma unroll
            for (int c = 0; c < H / 32; ++c) {
                tmem_wait_ld(r[c & 1]);
                // sign bits straight from the float sign bits (an exact ±0 needs e = 0,
                // i.e. a zero row, whose signs are all set below)
                uint32_t neg = 0u;
#pragma unroll
                for (int k = 31; k >= 0; --k) neg = __funnelshift_l(r[c & 1][k], neg, 1);
                sw[c] = n > 0.f ? ~neg : 0xffffffffu;
            }
            tc_fence_before();
            mbar_arrive(&sfree[slot]);
            if (live) {
                uint8_t* sd = signs + row * (int64_t)(D / 8) + half * (H / 8);
                if constexpr (H == 64) {
                    *reinterpret_cast<uint2*>(sd) = make_uint2(sw[0], sw[1]);
                } else {
                    *reinterpret_cast<uint32_t*>(sd) = sw[0];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

template <int D, int BM>
int launch_prod_tc(const tq_ctx& h, const CUtensorMap& tm_x, int64_t n_rows, const tq_planes& out, cudaStream_t s) {
    using C = ProdCfg<D>;
    static_assert(C::kSmemBytes <= 232448, "prod quantize shared memory above the per-CTA limit");
    auto fn = quantize_prod_tc_kernel<D, BM>;
    static std::atomic<uint64_t> smem_set{0};
    const int rc = ensure_smem_attr(smem_set, (const void*)fn, (int)C::kSmemBytes, "prod quantize smem attribute");
    if (rc != TQ_OK) return rc;
    const int64_t ntiles = (n_rows + kTile - 1) / kTile;
    const int grid = (int)(ntiles < h.num_sms ? ntiles : h.num_sms);
    const bool one = h.rot_passes == 1;
    fn<<<grid, kProdThreads, C::kSmemBytes, s>>>(tm_x, one ? h.dp.tm_pm : h.dp.tm_pi_hi, one ? h.dp.tm_pm : h.dp.tm_pi_lo,
                                                 h.dp.tm_t_hi, h.dp.tm_t_lo, n_rows, h.rot_passes, h.rot_norm_scale,
                                                 h.cb, out.codes, out.signs, out.norm, out.rnorm, h.dp.status);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "tensor-core prod quantize launch");
}

template <int D>
int launch_prod_tc_d(const tq_ctx& h, const CUtensorMap& tm_x, int64_t n_rows, const tq_planes& out, cudaStream_t s) {
    switch (h.hp.b_mse) {
        case 0: return launch_prod_tc<D, 0>(h, tm_x, n_rows, out, s);
        case 1: return launch_prod_tc<D, 1>(h, tm_x, n_rows, out, s);
        case 2: return launch_prod_tc<D, 2>(h, tm_x, n_rows, out, s);
        case 3: return launch_prod_tc<D, 3>(h, tm_x, n_rows, out, s);
        default: return fail(TQ_EUNSUPPORTED, "prod b_m=%d", h.hp.b_mse);
    }
}
// ---------------------------------------------------------------------------
// d = 256, prod: as the d = 256 mse path, Π is streamed with the row chunks, and
// so is T = SΠᵀ for the sketch.  Tensor memory holds one 512-column slot: Y (and,
// once read, the residual E as f16 hi/lo) in columns [0, 256), S = E·Tᵀ in
// [256, 512).  Per tile the ring carries four chunks of (X, Π_hi, Π_lo), then
// four chunks of (T_hi, T_lo); the MMA issuer runs MMA 1 over the first four,
// waits for the epilogue to write E, then MMA 2 over the next four (three f16
// passes, E read from tensor memory).  MMA 1 of the next tile overlaps the sign
// pass of this one.  Four epilogue warpgroups each take a 64-column quarter of
// every tile; the quarters' ‖y‖² and ‖e‖² meet in shared memory.
struct CfgP256 {
    static constexpr int D = 256;
    static constexpr int kChunks = D / kKC;                      // 4
    static constexpr int kXBytes = kTile * 128;                  // 16 KB
    static constexpr int kPBytes = D * 128;                      // 32 KB
    static constexpr int kStageBytes = kXBytes + 2 * kPBytes;    // 80 KB
    static constexpr size_t kBarOffset = (size_t)k256Stages * kStageBytes;
    static constexpr size_t kXchOffset = kBarOffset + 256;      // [2 sums][4 quarters][row]
    static constexpr size_t kSmemBytes = kXchOffset + (size_t)2 * 4 * kTile * 4 + 1024;
};

template <int BM>
__global__ void __launch_bounds__(k256Threads, 1)
quantize_prod_tc256_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_pi_hi,
                           const __grid_constant__ CUtensorMap tm_pi_lo, const __grid_constant__ CUtensorMap tm_t_hi,
                           const __grid_constant__ CUtensorMap tm_t_lo, int64_t n_rows, int npass, float norm_scale,
                           Codebook cb, uint8_t* __restrict__ codes, uint8_t* __restrict__ signs,
                           float* __restrict__ norm_out, float* __restrict__ rnorm_out, int* __restrict__ status) {
    using C = CfgP256;
    constexpr int D = C::D;
    constexpr int Q = D / 4;                    // columns per quarter
    constexpr int L = 1 << BM;
    constexpr int P = BM >= 1 ? L / 2 - 1 : 0;  // positive decision boundaries
    constexpr int WORDS = BM * D / 32;          // packed code words per row
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    allow_dependents();
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    uint64_t* full = bars;                 // [k256Stages] chunk landed
    uint64_t* empty = full + k256Stages;   // [k256Stages] chunk consumed by the MMAs
    uint64_t* yfull = empty + k256Stages;  // Y ready
    uint64_t* efull = yfull + 1;           // E written (512 arrivals)
    uint64_t* sfull = efull + 1;           // S ready
    uint64_t* sfree = sfull + 1;           // S read out (512 arrivals)
    uint64_t* drain = sfree + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = (n_rows + kTile - 1) / kTile;

    if (threadIdx.x == 0) {
        for (int s = 0; s < k256Stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(yfull, 1);
        mbar_init(efull, 512);
        mbar_init(sfull, 1);
        mbar_init(sfree, 512);
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ producer
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_pi_hi);
        prefetch_tensormap(&tm_pi_lo);
        prefetch_tensormap(&tm_t_hi);
        prefetch_tensormap(&tm_t_lo);
        int64_t q = 0;  // chunks issued
        bool ok = true;
        for (int64_t tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
            for (int c = 0; c < 2 * C::kChunks; ++c, ++q) {
                const int s = (int)(q % k256Stages);
                const int64_t u = q / k256Stages;
                if (u > 0 && !(ok = mbar_wait(&empty[s], (uint32_t)((u - 1) & 1), status, 31))) break;
                uint8_t* st = stages + (size_t)s * C::kStageBytes;
                if (c < C::kChunks) {  // X, Π_hi (, Π_lo) of chunk c
                    mbar_arrive_expect_tx(&full[s], C::kXBytes + npass * C::kPBytes);
                    tma_load_2d(st, &tm_x, &full[s], c * kKC, (int)(tile * kTile));
                    tma_load_2d(st + C::kXBytes, &tm_pi_hi, &full[s], c * kKC, 0);
                    if (npass == 2) tma_load_2d(st + C::kXBytes + C::kPBytes, &tm_pi_lo, &full[s], c * kKC, 0);
                } else {              // T_hi, T_lo of chunk c − 4
                    mbar_arrive_expect_tx(&full[s], 2 * C::kPBytes);
                    tma_load_2d(st + C::kXBytes, &tm_t_hi, &full[s], (c - C::kChunks) * kKC, 0);
                    tma_load_2d(st + C::kXBytes + C::kPBytes, &tm_t_lo, &full[s], (c - C::kChunks) * kKC, 0);
                }
            }
        }
        for (int64_t k = (q > k256Stages ? q - k256Stages : 0); k < q; ++k)
            mbar_wait(&full[k % k256Stages], (uint32_t)((k / k256Stages) & 1), status, 32);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc1 = idesc_bf16_f32(kTile, D);
        constexpr uint32_t idesc2 = idesc_f16_f32(kTile, D);
        const uint32_t base = smem_u32(stages);
        const uint32_t y_tmem = tmem_base, s_tmem = tmem_base + (uint32_t)D;
        int64_t q = 0, i = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++i) {
            // MMA 1: Y = X·Πᵀ into columns [0, D), once the previous tile's MMA 2 (which
            // reads E from these columns) has completed
            if (i > 0 && !(ok = mbar_wait(sfull, (uint32_t)((i - 1) & 1), status, 30))) break;
            for (int c = 0; c < C::kChunks; ++c, ++q) {
                const int s = (int)(q % k256Stages);
                if (!(ok = mbar_wait(&full[s], (uint32_t)((q / k256Stages) & 1), status, 33))) break;
                tc_fence_after();
                const uint32_t st = base + (uint32_t)(s * C::kStageBytes);
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    if (pass >= npass) break;
#pragma unroll
                    for (int kk = 0; kk < kKC / 16; ++kk) {
                        const uint64_t ad = smem_desc(st + kk * 32, 1024, 2);
                        const uint64_t bd = smem_desc(st + C::kXBytes + pass * C::kPBytes + kk * 32, 1024, 2);
                        mma_f16_ss(y_tmem, ad, bd, idesc1, (c | kk | pass) != 0);
                    }
                }
                mma_commit(&empty[s]);
            }
            if (!ok) break;
            mma_commit(yfull);
            // MMA 2: S = E·Tᵀ into columns [D, 2D), once the epilogue has written E and
            // has read the previous tile's S
            if (!(ok = mbar_wait(efull, (uint32_t)(i & 1), status, 34))) break;
            if (i > 0 && !(ok = mbar_wait(sfree, (uint32_t)((i - 1) & 1), status, 35))) break;
            tc_fence_after();
            for (int c = 0; c < C::kChunks; ++c, ++q) {
                const int s = (int)(q % k256Stages);
                if (!(ok = mbar_wait(&full[s], (uint32_t)((q / k256Stages) & 1), status, 36))) break;
                tc_fence_after();
                const uint32_t st = base + (uint32_t)(s * C::kStageBytes);
#pragma unroll
                for (int pass = 0; pass < 3; ++pass) {
#pragma unroll
                    for (int kk = 0; kk < kKC / 16; ++kk) {
                        const int k16 = 4 * c + kk;
                        // E_hi of dims 16·k16 … in columns 32·(k16/2) + 8·(k16%2), E_lo 16 columns further
                        const uint32_t acol = 32 * (k16 >> 1) + 8 * (k16 & 1) + (pass == 1 ? 16 : 0);
                        const uint64_t bd =
                            smem_desc(st + C::kXBytes + (pass == 2 ? C::kPBytes : 0) + kk * 32, 1024, 2);
                        mma_f16_ts(s_tmem, y_tmem + acol, bd, idesc2, (c | kk | pass) != 0);
                    }
                }
                mma_commit(&empty[s]);
            }
            if (!ok) break;
            mma_commit(sfull);
        }
        mma_commit(drain);
        mbar_wait(drain, 0, status, 37);
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue
        constexpr int GB = BM == 3 ? 24 : 16;  // bits per float packing group
        constexpr int GC = BM > 0 ? GB / BM : 1;
        constexpr int NG = BM > 0 ? 32 / GC : 1;
        constexpr float kAcc0 = (float)(1u << (GB - 1)) - 0.5f;
        const int qtr = (warp - 2) >> 2;        // quarter of the columns: 0..3
        const int quad = warp & 3;              // TMEM lane quadrant of this warp
        const int r_local = quad * 32 + lane;
        float* xss = reinterpret_cast<float*>(smem + C::kXchOffset);  // [quarter][row] partial ‖y‖²
        float* xes = xss + 4 * kTile;                                   // [quarter][row] partial ‖e‖²
        float t2[P > 0 ? P : 1];
#pragma unroll
        for (int p = 0; p < P; ++p) t2[p] = cb.t[L / 2 + p] * cb.t[L / 2 + p];
        CentroidPoly<BM> cp;
        cp.init(cb);
        const uint32_t lanebits = (uint32_t)(quad * 32) << 16;
        const uint32_t ybase = tmem_base + (uint32_t)(qtr * Q) + lanebits;
        const uint32_t sbase = ybase + (uint32_t)D;
        auto all_sync = [&]() { asm volatile("bar.sync 1, 512;" ::: "memory"); };
        // the quarters leave the tile loop together when a wait gives up
        auto all_ok = [&](bool ok) -> bool {
            uint32_t r;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\t"
                "setp.ne.u32 p, %1, 0;\n\t"
                "bar.red.and.pred q, 1, 512, p;\n\t"
                "selp.u32 %0, 1, 0, q;\n\t}\n"
                : "=r"(r)
                : "r"((uint32_t)ok)
                : "memory");
            return r != 0;
        };
        int64_t j = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++j) {
            if (!all_ok(mbar_wait(yfull, (uint32_t)(j & 1), status, 38))) break;
            tc_fence_after();
            uint32_t r[2][32];
            // pass 1: this quarter's part of ‖y‖², summed with the other quarters'
            uint64_t ss2 = 0ull;
            tmem_ld32(ybase, r[0]);
            tmem_ld32(ybase + 32, r[1]);
            tmem_wait_ld(r[0]);
            tmem_wait_ld(r[1]);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    const uint64_t v2 = f2(__uint_as_float(r[h][k]), __uint_as_float(r[h][k + 1]));
                    ss2 = fma2(v2, v2, ss2);
                }
            float ssa, ssb;
            f2_split(ss2, ssa, ssb);
            xss[qtr * kTile + r_local] = ssa + ssb;
            all_sync();
            const float ss = (xss[r_local] + xss[kTile + r_local]) + (xss[2 * kTile + r_local] + xss[3 * kTile + r_local]);
            const float n = sqrtf(ss);
            const float inv = n > 0.f ? 1.f / n : 0.f;
            const uint64_t inv2 = f2(inv, inv);
            const float cs = ss >= 0x1p-38f ? __fdividef(0x1p62f, ss) : 0x1p100f;
            const float kr = cs * ss;
            const uint64_t cs2 = f2(cs, cs);
            float kt2[P > 0 ? P : 1];
#pragma unroll
            for (int p = 0; p < P; ++p) kt2[p] = -kr * t2[p];
            const int64_t row = tile * kTile + r_local;
            const bool live = row < n_rows;
            const uint32_t keep = n == 0.f ? 0u : 0xffffffffu;
            const float live_f = n > 0.f ? 1.f : 0.f;
            uint64_t nc2[CentroidPoly<BM>::N];
#pragma unroll
            for (int k = 0; k < CentroidPoly<BM>::N; ++k) nc2[k] = f2(cp.m[k] * live_f, cp.m[k] * live_f);
            uint64_t es2 = 0ull;
            // pass 2: codes and the residual of this quarter's two 32-dim chunks (already in registers)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const uint32_t* rc = r[c];
                uint64_t acc[NG];
#pragma unroll
                for (int gi = 0; gi < NG; ++gi) acc[gi] = f2(kAcc0, 0.f);
                uint32_t ehi[16], elo[16];
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    const float va = __uint_as_float(rc[k]), vb = __uint_as_float(rc[k + 1]);
                    const uint64_t v2 = f2(va, vb);
                    uint64_t cnt2 = f2(0.5f, 0.5f);
                    if constexpr (P > 0) {
                        float wa, wb;
                        f2_split(mul2(v2, cs2), wa, wb);
#pragma unroll
                        for (int p = 0; p < P; ++p)
                            cnt2 = add2(cnt2, f2(__saturatef(fmaf(va, wa, kt2[p])), __saturatef(fmaf(vb, wb, kt2[p]))));
                    }
                    const uint32_t sga = __float_as_uint(va) & 0x80000000u, sgb = __float_as_uint(vb) & 0x80000000u;
                    uint64_t e2;
                    if constexpr (BM > 0) {
                        float ca, cb2;
                        f2_split(cnt2, ca, cb2);
                        const float sa = __uint_as_float(__float_as_uint(ca) | sga);
                        const float sb = __uint_as_float(__float_as_uint(cb2) | sgb);
                        acc[k / GC] = fma2(f2(sa, sb),
                                           f2((float)(1u << (BM * (k % GC))), (float)(1u << (BM * ((k + 1) % GC)))),
                                           acc[k / GC]);
                        // residual e = sign(y)·(|y|/‖y‖ − c⁺(count)) (0 for a zero row)
                        constexpr int N = CentroidPoly<BM>::N;
                        uint64_t nc = nc2[N - 1];
#pragma unroll
                        for (int qq = N - 2; qq >= 0; --qq) nc = fma2(nc, cnt2, nc2[qq]);
                        float ta, tb;
                        f2_split(fma2(f2(fabsf(va), fabsf(vb)), inv2, nc), ta, tb);
                        e2 = f2(__uint_as_float(__float_as_uint(ta) ^ sga), __uint_as_float(__float_as_uint(tb) ^ sgb));
                    } else {
                        e2 = mul2(v2, inv2);
                    }
                    es2 = fma2(e2, e2, es2);
                    float ea, eb;
                    f2_split(e2, ea, eb);
                    const __half2 hi = __floats2half2_rn(ea, eb);
                    const float2 hf = __half22float2(hi);
                    const __half2 lo = __floats2half2_rn(ea - hf.x, eb - hf.y);
                    ehi[k / 2] = *reinterpret_cast<const uint32_t*>(&hi);
                    elo[k / 2] = *reinterpret_cast<const uint32_t*>(&lo);
                }
                // the residual of these 32 dims replaces their (already read) Y columns
                tmem_st16(ybase + c * 32, ehi);
                tmem_st16(ybase + c * 32 + 16, elo);
                if constexpr (BM > 0) {
                    uint32_t cw[BM];
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
                    if (live) {
                        uint8_t* cd = codes + row * (int64_t)(WORDS * 4) + (qtr * (Q / 32) + c) * (BM * 4);
                        if constexpr (BM == 2) {
                            *reinterpret_cast<uint2*>(cd) = make_uint2(cw[0] & keep, cw[1] & keep);
                        } else {
#pragma unroll
                            for (int w = 0; w < BM; ++w) reinterpret_cast<uint32_t*>(cd)[w] = cw[w] & keep;
                        }
                    }
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(efull);
            float esa, esb;
            f2_split(es2, esa, esb);
            xes[qtr * kTile + r_local] = esa + esb;
            all_sync();
            if (live && qtr == 0) {
                norm_out[row] = n * norm_scale;
                rnorm_out[row] = sqrtf((xes[r_local] + xes[kTile + r_local]) + (xes[2 * kTile + r_local] + xes[3 * kTile + r_local]));
            }
            // pass 3: sign bits of this quarter of S = T·e (bit i set ⇔ s_i ≥ 0)
            if (!all_ok(mbar_wait(sfull, (uint32_t)(j & 1), status, 39))) break;
            tc_fence_after();
            tmem_ld32(sbase, r[0]);
            tmem_ld32(sbase + 32, r[1]);
            tmem_wait_ld(r[0]);
            tmem_wait_ld(r[1]);
            tc_fence_before();
            mbar_arrive(sfree);
            uint32_t sw[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t neg = 0u;
#pragma unroll
                for (int k = 31; k >= 0; --k) neg = __funnelshift_l(r[c][k], neg, 1);
                sw[c] = n > 0.f ? ~neg : 0xffffffffu;
            }
            if (live) *reinterpret_cast<uint2*>(signs + row * (int64_t)(D / 8) + qtr * (Q / 8)) = make_uint2(sw[0], sw[1]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

template <int BM>
int launch_prod_tc256(const tq_ctx& h, const CUtensorMap& tm_x, int64_t n_rows, const tq_planes& out,
                      cudaStream_t s) {
    using C = CfgP256;
    static_assert(C::kSmemBytes <= 232448, "d = 256 prod quantize shared memory above the per-CTA limit");
    auto fn = quantize_prod_tc256_kernel<BM>;
    static std::atomic<uint64_t> smem_set{0};
    const int rc = ensure_smem_attr(smem_set, (const void*)fn, (int)C::kSmemBytes, "d=256 prod quantize smem attribute");
    if (rc != TQ_OK) return rc;
    const int64_t ntiles = (n_rows + kTile - 1) / kTile;
    const int grid = (int)(ntiles < h.num_sms ? ntiles : h.num_sms);
    const bool one = h.rot_passes == 1;
    fn<<<grid, k256Threads, C::kSmemBytes, s>>>(tm_x, one ? h.dp.tm_pm : h.dp.tm_pi_hi, one ? h.dp.tm_pm : h.dp.tm_pi_lo,
                                                h.dp.tm_t_hi, h.dp.tm_t_lo, n_rows, h.rot_passes, h.rot_norm_scale, h.cb,
                                                out.codes, out.signs, out.norm, out.rnorm, h.dp.status);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "d=256 tensor-core prod quantize launch");
}

int launch_prod_tc256_b(const tq_ctx& h, const CUtensorMap& tm_x, int64_t n_rows, const tq_planes& out,
                        cudaStream_t s) {
    switch (h.hp.b_mse) {
        case 0: return launch_prod_tc256<0>(h, tm_x, n_rows, out, s);
        case 1: return launch_prod_tc256<1>(h, tm_x, n_rows, out, s);
        case 2: return launch_prod_tc256<2>(h, tm_x, n_rows, out, s);
        case 3: return launch_prod_tc256<3>(h, tm_x, n_rows, out, s);
        default: return fail(TQ_EUNSUPPORTED, "prod b_m=%d", h.hp.b_mse);
    }
}

// One CTA whose pipeline wait nothing completes: the bounded wait gives up after
// limit_ns, records `code` in the status word and the kernel returns.  It checks
// the failure path of every pipeline in this file without faulting anything.
__global__ void expire_wait_kernel(int* status, int code, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, status, code, limit_ns);
    __syncthreads();
}

}  // namespace

int launch_expire_wait(const tq_ctx& h, int code, uint64_t limit_ns, cudaStream_t s) {
    expire_wait_kernel<<<1, 32, 0, s>>>(h.dp.status, code, limit_ns);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "wait-timeout check launch");
}

bool quantize_tc_supported(const tq_ctx& h, int x_dtype, int64_t n_rows) {
    // TMA row coordinates are 32-bit signed: the last tile must start below 2^31.
    const bool rot = h.rot_passes == 1 ? h.dp.Pm != nullptr : h.dp.Pi_hi != nullptr;
    const bool params = h.hp.variant == TQ_MSE ? rot : (rot && h.dp.T_hi != nullptr && h.hp.b_mse <= 3);
    const bool dim = h.hp.d == 64 || h.hp.d == 128 || h.hp.d == 256;
    const bool f32 = x_dtype == TQ_F32 && h.hp.variant == TQ_MSE && (h.hp.d == 64 || h.hp.d == 128);
    return (x_dtype == TQ_BF16 || f32) && dim && params && h.num_sms > 0 && n_rows < ((int64_t)1 << 31) - kTile;
}

bool quantize_pair_tc_supported(const tq_ctx& ha, const tq_ctx& hb, int x_dtype, int64_t rows_a, int64_t rows_b) {
    return ha.hp.variant == TQ_MSE && hb.hp.variant == TQ_MSE && ha.hp.d == hb.hp.d && (ha.hp.d == 64 || ha.hp.d == 128) &&
           ha.hp.b_mse == hb.hp.b_mse && ha.rot_passes == hb.rot_passes && rows_a > 0 && rows_b > 0 &&
           quantize_tc_supported(ha, x_dtype, rows_a) && quantize_tc_supported(hb, x_dtype, rows_b) &&
           ha.num_sms == hb.num_sms;
}

int launch_quantize_pair_tc(const tq_ctx& ha, const void* xa, int64_t rows_a, int64_t stride_a, const tq_planes& out_a,
                            const tq_ctx& hb, const void* xb, int64_t rows_b, int64_t stride_b, const tq_planes& out_b,
                            int x_dtype, cudaStream_t s) {
    const int d = ha.hp.d;
    if (x_dtype == TQ_F32) {
        const TcSide a = make_side(ha, nullptr, static_cast<const float*>(xa), stride_a, rows_a, out_a);
        const TcSide b = make_side(hb, nullptr, static_cast<const float*>(xb), stride_b, rows_b, out_b);
        return d == 64 ? launch_tc_pair_d<64, true>(ha.hp.b_mse, a, b, ha.rot_passes, ha.num_sms, s)
                       : launch_tc_pair_d<128, true>(ha.hp.b_mse, a, b, ha.rot_passes, ha.num_sms, s);
    }
    CUtensorMap ma, mb;
    int rc = encode_tmap_bf16_2d(&ma, xa, (uint64_t)d, (uint64_t)rows_a, (uint64_t)stride_a * 2, kKC, kTile);
    if (rc != TQ_OK) return rc;
    rc = encode_tmap_bf16_2d(&mb, xb, (uint64_t)d, (uint64_t)rows_b, (uint64_t)stride_b * 2, kKC, kTile);
    if (rc != TQ_OK) return rc;
    const TcSide a = make_side(ha, &ma, nullptr, 0, rows_a, out_a);
    const TcSide b = make_side(hb, &mb, nullptr, 0, rows_b, out_b);
    return d == 64 ? launch_tc_pair_d<64, false>(ha.hp.b_mse, a, b, ha.rot_passes, ha.num_sms, s)
                   : launch_tc_pair_d<128, false>(ha.hp.b_mse, a, b, ha.rot_passes, ha.num_sms, s);
}

int launch_quantize_tc(const tq_ctx& h, const void* x, int x_dtype, int64_t n_rows, int64_t stride,
                       const tq_planes& out, cudaStream_t s) {
    if (x_dtype == TQ_F32) {
        const float* xf = static_cast<const float*>(x);
        return h.hp.d == 64 ? launch_tc_f32_d<64>(h, xf, n_rows, stride, out, s)
                            : launch_tc_f32_d<128>(h, xf, n_rows, stride, out, s);
    }
    CUtensorMap tm_x;
    int rc = encode_tmap_bf16_2d(&tm_x, x, (uint64_t)h.hp.d, (uint64_t)n_rows, (uint64_t)stride * 2, kKC, kTile);
    if (rc != TQ_OK) return rc;
    const bool prod = h.hp.variant == TQ_PROD;
    switch (h.hp.d) {
        case 64: return prod ? launch_prod_tc_d<64>(h, tm_x, n_rows, out, s) : launch_tc_d<64>(h, tm_x, n_rows, out, s);
        case 128:
            return prod ? launch_prod_tc_d<128>(h, tm_x, n_rows, out, s) : launch_tc_d<128>(h, tm_x, n_rows, out, s);
        case 256:
            return prod ? launch_prod_tc256_b(h, tm_x, n_rows, out, s) : launch_tc256_b(h, tm_x, n_rows, out, s);
        default: return fail(TQ_EUNSUPPORTED, "tensor-core quantize: d=%d", h.hp.d);
    }
}

}  // namespace tq
