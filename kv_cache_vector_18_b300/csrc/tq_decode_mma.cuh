// Split-K decode attention over the packed cache on the tensor cores, d = 128.
//
// Same computation as the CUDA-core split kernel (see tq_decode.cu and
// include/tq.h): per (batch, KV head, head block of 8 query heads, token chunk)
// an online softmax over
//   s_t = scale·‖k_t‖·(⟨q′, c_k[code_t]⟩ + √(π/2)/d·‖r_t‖·⟨q″, z_t⟩)
// and a value sum in the rotated frame, Σ_t p_t·‖v_t‖·c_v[code_t] (+ the QJL
// part for prod values), written as one split partial (m, l, acc) per head.
//
// Mapping onto mma.sync.m16n8k16 (f16 operands, f32 accumulators), per warp and
// 16-token step made of two 8-token groups, lane = 4·g + c:
//   scores  S[16 × 8 tokens] = [Q′_hi; Q′_lo][16 × d] · K̃ᵀ[d × 8 tokens]: the keys
//           are the B operand, so rows 0–7 (f16 high parts of the 8 heads' q′)
//           and rows 8–15 (their f16 rounding errors) use the whole M = 16 and
//           the score keeps ~2⁻²² of q′ at no extra MMA.  Lane (g, c) decodes
//           token g of the group: for k16 block kb its B fragment is four
//           consecutive codes of the token's row (one byte at 2 bits: one 64-bit
//           load from a table of code quads; two code-pair loads at 3 and 4
//           bits; two bit operations per pair at 1 bit).
//   QJL     Z·Q″ᵀ in the same orientation, [Q″_hi; Q″_lo] · Zᵀ: one byte of sign
//           bits gives the ±1 fragments of two k16 blocks through one 128-bit
//           table load.
//   values  Oᵀ[d × 8 heads] += Ṽᵀ[d × 16 tokens] · P′ᵀ[16 × 8]: Ṽ is decoded
//           token-major (code-pair tables) and moved to the dim-major A layout
//           with movmatrix.trans; P′ leaves the score accumulator already in the
//           B-fragment layout (lane (g, c): head g, tokens 2c, 2c + 1 of each group).
// Each lane keeps the online-softmax state of one head (g).  ‖v_t‖ is folded
// into the softmax exponent (P′_t = 2^(s_t·log2e + log2‖v_t‖ − M)), so the f16
// weights stay bounded whatever the value norms; l accumulates P′_t/‖v_t‖ in f32
// against the same running maximum M.  M is raised only when a step's exponent
// exceeds it by more than kSlack, so P′ ≤ 2^kSlack and most steps skip the
// cross-lane maximum.  Per-head scale factors keep the f16 query fragments in
// [−1, 1], and the centroid tables hold f16(σ·c) for a per-codebook σ chosen on
// the host so that the f16 rounding of the centroids — systematic, and
// amplified by the softmax — nearly vanishes.
//
// Data movement: one producer warp streams the chunk's packed planes into a
// ring of shared-memory stages of 64 or 128 tokens (one bulk copy per plane and stage,
// or per-lane cp.async when the slab's norm rows are not 16-byte aligned), each
// stage completing on a "full" mbarrier; the consumer warps prepare tables and
// queries meanwhile (synchronising among themselves only), then take 16-token
// tiles of the stages round-robin, read their operands with short shared-memory
// loads and release each stage on an "empty" mbarrier (every wait is bounded).
// The last CTA of each (batch, KV head, head block) to finish merges every
// split's partial and applies Π_vᵀ on the tensor cores (no merge launch).
//
// Variants (kernel template flags): with at most four query heads per KV head
// (G4) the scores and QJL sums take the keys and signs as the A operand instead
// (step4: one MMA per k16 block for the 16 tokens), and a CTA whose chunk lies
// past its sequence's length skips its staging and prologue; behind the
// decode-step append with long chunks (AA) the CTA streams the rows below the
// pre-append length before waiting for the append.
#pragma once

#include <math.h>

#include "tq_common.cuh"
#include "tq_decode_args.h"
#include "tq_sm100.cuh"

namespace tq {
namespace mmadec {

constexpr int D = 128;
constexpr int kHeads = 8;   // query heads per CTA: one n8 MMA tile
constexpr int kTile = 16;   // tokens per warp step
constexpr int kKB = D / 16; // k16 blocks of the score contraction
constexpr int kMT = D / 16; // m16 tiles of the value contraction
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kSlack = 8.f; // log2 headroom before the running maximum is raised

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma16816_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8×8 b16 tile held one row-pair per lane (fragment layout).
__device__ __forceinline__ uint32_t mov_trans(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Rotated queries in shared memory: each head's 128 values as four 32-value
// chunks padded to 36, so that lane (g, c) reading chunk c of head g with 16-byte
// loads never collides on a bank with the other lanes of its quarter-warp.
constexpr int kQChunk = 36;
constexpr int kQRow = 4 * kQChunk;
__host__ __device__ constexpr int qidx(int h, int j) { return h * kQRow + (j >> 5) * kQChunk + (j & 31); }

// ---- 8 heads × a d × d matrix on mma.sync with bf16 hi/lo operands ------------
// r[h][i] = Σ_j M[i][j]·x[h][j] for a matrix held as M = M_hi + M_lo (bf16,
// row-major [i][j]) and fp32 rows x.  The A operand is [x_hi; x_lo] (rows g and
// g + 8 of the MMA), so the two halves of each output come out in rows g and g + 8
// and their sum carries fp32-level accuracy.  The contraction order is permuted so
// that in k16 blocks 2p and 2p + 1 lane (g, c) holds the eight consecutive dims
// 32p + 8c … 32p + 8c + 7: its matrix operand is one 16-byte load of row i0 + g.
// A fragments of head g from its fp32 row xg (dims contiguous).
__device__ __forceinline__ void hilo_a(const float* xg, int c, uint32_t (&A)[kKB][4]) {
#pragma unroll
    for (int ks = 0; ks < kKB; ++ks)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int d0 = 32 * (ks >> 1) + 8 * c + 4 * (ks & 1) + 2 * hh;
            const float2 x = *reinterpret_cast<const float2*>(xg + d0);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(x.x, x.y);
            const float2 hf = __bfloat1622float2(hi);
            A[ks][2 * hh] = *reinterpret_cast<const uint32_t*>(&hi);
            A[ks][2 * hh + 1] = pack_bf2(x.x - hf.x, x.y - hf.y);
        }
}
// The same from a bf16 row: x is exact in bf16, so the low rows are zero.
__device__ __forceinline__ void hilo_a(const __nv_bfloat16* xg, int c, uint32_t (&A)[kKB][4]) {
#pragma unroll
    for (int ks = 0; ks < kKB; ++ks)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int d0 = 32 * (ks >> 1) + 8 * c + 4 * (ks & 1) + 2 * hh;
            A[ks][2 * hh] = *reinterpret_cast<const uint32_t*>(xg + d0);
            A[ks][2 * hh + 1] = 0u;
        }
}
// this lane's 16-byte pieces of rows i0 + g of M_hi and M_lo
__device__ __forceinline__ void hilo_b(const uint16_t* Mhi, const uint16_t* Mlo, int i0, int g, int c,
                                       uint4 (&bh)[kKB / 2], uint4 (&bl)[kKB / 2]) {
    const int row = ((i0 + g) * D + 8 * c) >> 3;  // 16-byte index of (i0 + g, 8c)
#pragma unroll
    for (int p2 = 0; p2 < kKB / 2; ++p2) {
        bh[p2] = __ldg(reinterpret_cast<const uint4*>(Mhi) + row + 4 * p2);
        bl[p2] = __ldg(reinterpret_cast<const uint4*>(Mlo) + row + 4 * p2);
    }
}
__device__ __forceinline__ void hilo_mma(float (&acc)[4], const uint32_t (&A)[kKB][4], const uint4 (&bh)[kKB / 2],
                                         const uint4 (&bl)[kKB / 2]) {
#pragma unroll
    for (int ks = 0; ks < kKB; ++ks) {
        const uint4 h = bh[ks >> 1], l = bl[ks >> 1];
        mma16816_bf16(acc, A[ks], (ks & 1) ? h.z : h.x, (ks & 1) ? h.w : h.y);
        mma16816_bf16(acc, A[ks], (ks & 1) ? l.z : l.x, (ks & 1) ? l.w : l.y);
    }
}

// Bits [bit, bit + NBITS) of the little-endian word run w, returned shifted
// left by S0 (a byte offset into a table whose entries are 2^S0 bytes apart).
template <int NBITS, int S0>
__device__ __forceinline__ uint32_t field_off(const uint32_t* w, int bit) {
    const int wi = bit >> 5, sh = bit & 31;
    uint32_t x;
    if (sh >= S0) {
        if (sh + NBITS <= 32)
            x = w[wi] >> (sh - S0);
        else
            x = __funnelshift_r(w[wi], w[wi + 1], sh - S0);
    } else {
        x = w[wi] << (S0 - sh);
    }
    return x & (((1u << NBITS) - 1u) << S0);
}

// 32-bit shared-memory load at a byte address (kept separate so that each
// result can be placed straight into its MMA operand register).
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
template <int OFF>
__device__ __forceinline__ uint32_t lds32o(uint32_t addr) {
    uint32_t v;
    asm("ld.shared.b32 %0, [%1+%2];" : "=r"(v) : "r"(addr), "n"(OFF));
    return v;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// cp.async of 16 (or 4) bytes; src_bytes = 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int OFF>
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm("ld.shared.v2.b32 {%0, %1}, [%2+%3];" : "=r"(v.x), "=r"(v.y) : "r"(addr), "n"(OFF));
    return v;
}

// A ±1 (or ±c) f16 pair from two bits of w that are 16 apart: bits τ and τ + 16
// land in the two sign positions and flip the pair `neg` (whose halves are
// negative) where they are set.
__device__ __forceinline__ uint32_t flip_pair(uint32_t w, int tau, uint32_t neg) {
    return neg ^ ((w << (15 - tau)) & 0x80008000u);
}

constexpr uint32_t kMinusOnePair = 0xBC00BC00u;  // f16 (−1, −1)

// Every table sits at a shared-memory address that is a multiple of its
// (power-of-two) size, so a lookup address is one OR of the shifted code field
// with the lane's copy offset and the table base.  Table layouts (σ = the
// codebook's table scale):
//   quad (b = 2): entry e (a byte: four 2-bit codes, LSB first) holds the two f16
//          pairs (σc[e₀], σc[e₁]), (σc[e₂], σc[e₃]) as 8 bytes, 16 copies
//          (128-byte entries), so a half-warp's 64-bit loads never collide;
//   pair (b = 3, 4): entry e (two b-bit codes) holds (σc[e₀], σc[e₁]), 32 copies.
template <int B>
struct Table {
    static constexpr bool kQuad = B == 2;
    static constexpr bool kPair = B >= 3;
    static constexpr size_t kBytes =
        kPair ? (size_t)(1 << (2 * B)) * 32 * 4 : (kQuad ? (size_t)256 * 16 * 8 : 0);
    // Filled by nt threads (thread tid; nt and the entry counts multiples of 32, so
    // whole warps take part in each round).  Lane k holds centroid k, and an
    // entry's centroids come from shuffles: indexing the parameter codebook with
    // per-lane indices would serialise constant-cache reads.
    __device__ static void fill(unsigned char* tabp, const Codebook& cb, int tid, int nt) {
        const int lane = tid & 31;
        float cl = 0.f;
#pragma unroll
        for (int k = 0; k < (1 << B); ++k)
            if (lane == k) cl = cb.c[k] * cb.lut_scale;
        if constexpr (kQuad) {
            for (int i = tid; i < 256 * 16; i += nt) {
                const uint32_t e = (uint32_t)i >> 4, copy = (uint32_t)i & 15u;
                const float c0 = __shfl_sync(0xffffffffu, cl, (int)(e & 3)), c1 = __shfl_sync(0xffffffffu, cl, (int)((e >> 2) & 3));
                const float c2 = __shfl_sync(0xffffffffu, cl, (int)((e >> 4) & 3)), c3 = __shfl_sync(0xffffffffu, cl, (int)((e >> 6) & 3));
                *reinterpret_cast<uint2*>(tabp + e * 128u + copy * 8u) = make_uint2(pack_h2(c0, c1), pack_h2(c2, c3));
            }
        }
        if constexpr (kPair) {
            constexpr uint32_t m = (1u << B) - 1u;
            for (int i = tid; i < (1 << (2 * B)) * 32; i += nt) {
                const uint32_t e = (uint32_t)i >> 5, copy = (uint32_t)i & 31u;
                const float c0 = __shfl_sync(0xffffffffu, cl, (int)(e & m));
                const float c1 = __shfl_sync(0xffffffffu, cl, (int)((e >> B) & m));
                *reinterpret_cast<uint32_t*>(tabp + e * 128u + copy * 4u) = pack_h2(c0, c1);
            }
        }
    }
    // this lane's view of the table (base | copy offset)
    __device__ static uint32_t lane_base(const unsigned char* tabp, int lane) {
        return smem_addr(tabp) + (kQuad ? (uint32_t)(lane & 15) * 8u : (uint32_t)lane * 4u);
    }
};

// ---- keys: the B operand of the score MMA ------------------------------------
// Lane (g, c) decodes token g of an 8-token group from its run of 32 codes
// (dims [32c, 32c + 32), KB words starting at byte 4·KB·c of the row).  For k16
// block kb the fragment (b0, b1) holds, in MMA k slots 2c, 2c + 1, 2c + 8,
// 2c + 9, the dims dim(c, kb, 0..3); the Q′ fragments follow the same map.
//   KB = 1: pairs of bits 16 apart, (2kb, 2kb + 16) and (2kb + 1, 2kb + 17):
//           the centroids are ±c₁, two bit operations per pair;
//   KB = 2: byte kb of the run, one 64-bit load from the quad table;
//   KB = 3, 4: codes 4kb … 4kb + 3 of the run, two loads from the pair table.
template <int KB>
struct KDecoder {
    uint32_t k0;   // KB = 1: (−σc₁, −σc₁)
    uint32_t tab;  // KB ≥ 2: table base | lane copy offset
    __device__ void init(const Codebook& cb, const unsigned char* tabp, int lane) {
        if constexpr (KB == 1) k0 = pack_h2(cb.c[0] * cb.lut_scale, cb.c[0] * cb.lut_scale);
        if constexpr (KB >= 2) tab = Table<KB>::lane_base(tabp, lane);
    }
    __device__ __forceinline__ void frag(const uint32_t* w, int kb, uint32_t& b0, uint32_t& b1) const {
        if constexpr (KB == 1) {
            b0 = flip_pair(w[0], 2 * kb, k0);
            b1 = flip_pair(w[0], 2 * kb + 1, k0);
        } else if constexpr (KB == 2) {
            const uint2 v = lds64<0>(field_off<8, 7>(w, 8 * kb) | tab);
            b0 = v.x;
            b1 = v.y;
        } else {
            b0 = lds32(field_off<2 * KB, 7>(w, 4 * KB * kb) | tab);
            b1 = lds32(field_off<2 * KB, 7>(w, 4 * KB * kb + 2 * KB) | tab);
        }
    }
    __host__ __device__ static constexpr int dim(int c, int kb, int e) {
        return KB == 1 ? 32 * c + 2 * kb + (e >> 1) + 16 * (e & 1) : 32 * c + 4 * kb + e;
    }
};

// QJL signs of the keys: word c of a token's sign row holds dims [32c, 32c + 32);
// byte j of it (eight signs, LSB first) gives the fragments of k16 blocks 2j and
// 2j + 1 through one 128-bit load from a table whose entry e holds the four f16
// ±1 pairs of e's bits (0, 1), (2, 3), (4, 5), (6, 7) — (b0, b1) of block 2j,
// then (b0, b1) of block 2j + 1.  Eight copies (128-byte entries) keep each
// quarter-warp's loads apart.  Block kb covers dims 32c + 4kb … 32c + 4kb + 3.
struct KSignTable {
    static constexpr size_t kBytes = (size_t)256 * 8 * 16;
    __device__ static void fill(unsigned char* tabp, int tid, int nt) {
        for (int i = tid; i < 256 * 8; i += nt) {
            const uint32_t e = (uint32_t)i >> 3, copy = (uint32_t)i & 7u;
            uint32_t v[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const uint32_t lo = (e >> (2 * p)) & 1u ? 0x3C00u : 0xBC00u;
                const uint32_t hi = (e >> (2 * p + 1)) & 1u ? 0x3C00u : 0xBC00u;
                v[p] = lo | (hi << 16);
            }
            *reinterpret_cast<uint4*>(tabp + e * 128u + copy * 16u) = make_uint4(v[0], v[1], v[2], v[3]);
        }
    }
    __device__ static uint32_t lane_base(const unsigned char* tabp, int lane) {
        return smem_addr(tabp) + (uint32_t)(lane & 7) * 16u;
    }
};
__host__ __device__ constexpr int ksign_dim(int c, int kb, int e) { return 32 * c + 4 * kb + e; }

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// ---- values: token-major pairs for movmatrix ----------------------------------
// A lane owns a run of 32 consecutive codes of a row (dims [32c, 32c + 32)).
// Decoder<B>::pairs(w, m, p0, p1) yields the two f16 pairs that m16 tile m of
// the value operand takes from that run (pairs τ = 2m and 2m + 1, before the
// transpose), and Decoder<B>::dim(c, τ, e) is the dim held by element e of pair
// τ — the accumulator rows follow the same map.
//   B = 1: both codes of a pair are bits τ and τ + 16 of the run's word (±c₁).
//   B = 2: byte m of the run, one 64-bit load from the quad table.
//   B = 3, 4: two adjacent codes per pair, one load each from the pair table.
template <int B>
struct Decoder {
    static constexpr size_t kTableBytes = Table<B>::kBytes;
    uint32_t k0;
    uint32_t tab;
    __device__ void init(const Codebook& cb, const unsigned char* tabp, int lane) {
        if constexpr (B == 1) k0 = pack_h2(cb.c[0] * cb.lut_scale, cb.c[0] * cb.lut_scale);
        if constexpr (B >= 2) tab = Table<B>::lane_base(tabp, lane);
    }
    __device__ __forceinline__ void pairs(const uint32_t* w, int kb, uint32_t& p0, uint32_t& p1) const {
        if constexpr (B == 1) {
            p0 = flip_pair(w[0], 2 * kb, k0);
            p1 = flip_pair(w[0], 2 * kb + 1, k0);
        } else if constexpr (B == 2) {
            const uint2 v = lds64<0>(field_off<8, 7>(w, 8 * kb) | tab);
            p0 = v.x;
            p1 = v.y;
        } else {
            p0 = lds32(field_off<2 * B, 7>(w, 4 * B * kb) | tab);
            p1 = lds32(field_off<2 * B, 7>(w, 4 * B * kb + 2 * B) | tab);
        }
    }
    __host__ __device__ static constexpr int dim(int c, int tau, int e) {
        return B == 1 ? 32 * c + tau + 16 * e : 32 * c + 2 * tau + e;
    }
};

// QJL sign pairs of the values (prod values): pair τ of a lane's sign word is
// bits (τ, τ + 16), two bit operations each; quad(w, m, p) gives pairs 4m … 4m + 3.
struct SignDecoder {
    __device__ __forceinline__ void quad(uint32_t w, int m, uint32_t (&p)[4]) const {
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = flip_pair(w, 4 * m + i, kMinusOnePair);
    }
    __host__ __device__ static constexpr int dim(int c, int tau, int e) { return 32 * c + tau + 16 * e; }
};
__host__ __device__ constexpr int sign_dim(int c, int tau, int e) { return SignDecoder::dim(c, tau, e); }

// Tokens per stage of the CTA's staging ring (four 16-token tiles), and the
// most stages a ring holds (it takes what shared memory the tables leave).
constexpr int kStageRows = 64;
// With QJL planes (six or eight bulk copies per stage) stages are 128 tokens, so
// that the producer's one issuing lane keeps ahead of the consumers.
template <bool KP, bool VP>
constexpr int stage_rows() { return KP || VP ? 2 * kStageRows : kStageRows; }
constexpr int kMaxStages = 12;

// Byte layout of one stage (R tokens) of every plane: plane by plane,
// rows in token order, so a 16-token tile of a plane is one contiguous run.
template <int KB, bool KP, int VB, bool VP>
struct Stage {
    static constexpr int R = stage_rows<KP, VP>();
    static constexpr int kRK = KB * 16, kRV = VB * 16;  // code bytes per row
    static constexpr int kKC = 0;
    static constexpr int kKS = kKC + R * kRK;
    static constexpr int kKN = kKS + (KP ? R * 16 : 0);
    static constexpr int kKR = kKN + R * 4;
    static constexpr int kVC = kKR + (KP ? R * 4 : 0);
    static constexpr int kVS = kVC + R * kRV;
    static constexpr int kVN = kVS + (VP ? R * 16 : 0);
    static constexpr int kVR = kVN + R * 4;
    static constexpr int kBytes = kVR + (VP ? R * 4 : 0);
};

// Plane pointers of this CTA's (batch, KV head) slab.
struct Slab {
    bool a16;  // the slab's norm planes start on a 16-byte boundary
    const uint8_t* kc;
    const uint8_t* ks;
    const float* kn;
    const float* krn;
    const uint8_t* vc;
    const uint8_t* vs;
    const float* vn;
    const float* vrn;
};

// The producer warp's copy of one stage: rows [tb, tb + valid) of every plane of
// the slab into the stage at dst with per-lane cp.async; rows from `valid` to
// the stage's R are zero-filled and nothing past the chunk's last token is read.
template <int RB, int R>  // bytes per row (a multiple of 16), rows per stage
__device__ __forceinline__ void copy_rows16(uint32_t dst, const uint8_t* src, int valid, int lane) {
    constexpr int kChunks = R * RB / 16, kPerRow = RB / 16;
#pragma unroll
    for (int r = 0; r < (kChunks + 31) / 32; ++r) {
        const int q = lane + 32 * r;
        if (kChunks % 32 == 0 || q < kChunks) {
            const bool ok = q / kPerRow < valid;
            cp_async16(dst + 16 * q, ok ? src + 16 * q : src, ok ? 16u : 0u);
        }
    }
}
// fp32 norms: 16-byte chunks of four rows when the plane's rows start on a
// 16-byte boundary (a16), else one 4-byte copy per row
template <int R>
__device__ __forceinline__ void copy_norms(uint32_t dst, const float* src, bool a16, int valid, int lane) {
    if (a16) {
#pragma unroll
        for (int q = lane; q < R / 4; q += 32) {
            const int n = min(4, max(0, valid - 4 * q));
            cp_async16(dst + 16 * q, n > 0 ? src + 4 * q : src, 4u * (uint32_t)n);
        }
    } else {
#pragma unroll
        for (int i = lane; i < R; i += 32) {
            const bool ok = i < valid;
            cp_async4(dst + 4 * i, ok ? src + i : src, ok ? 4u : 0u);
        }
    }
}

// Bulk variant (T_max % 4 == 0): rows [tb, tb + min(R, T_max − tb)) of
// every plane with one untiled bulk copy each, completing on the stage's full
// mbarrier.  The row count is a multiple of 4, so every copy is a multiple of 16
// bytes and starts on a 16-byte boundary; rows past the chunk's end are masked
// in the step, and nothing past the slab is read.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

template <int KB, bool KP, int VB, bool VP>
__device__ __forceinline__ void produce_stage_bulk(uint32_t dst, uint32_t bar, const Slab& s, int tb, int T_max) {
    using ST = Stage<KB, KP, VB, VP>;
    // bytes of one row over all planes: codes, norms (keys and values), signs and residual norms
    constexpr uint32_t kRowBytes = ST::kRK + ST::kRV + 8 + (KP ? 20 : 0) + (VP ? 20 : 0);
    static_assert(kRowBytes * ST::R == ST::kBytes, "bulk staging must fill the whole stage layout");
    const uint32_t rows = (uint32_t)min(ST::R, T_max - tb);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the consumers' reads of the slot come first
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(rows * kRowBytes)
                 : "memory");
    if constexpr (KB > 0) bulk_g2s(dst + ST::kKC, s.kc + (size_t)tb * ST::kRK, rows * ST::kRK, bar);
    if constexpr (KP) {
        bulk_g2s(dst + ST::kKS, s.ks + (size_t)tb * 16, rows * 16, bar);
        bulk_g2s(dst + ST::kKR, s.krn + tb, rows * 4, bar);
    }
    bulk_g2s(dst + ST::kKN, s.kn + tb, rows * 4, bar);
    if constexpr (VB > 0) bulk_g2s(dst + ST::kVC, s.vc + (size_t)tb * ST::kRV, rows * ST::kRV, bar);
    if constexpr (VP) {
        bulk_g2s(dst + ST::kVS, s.vs + (size_t)tb * 16, rows * 16, bar);
        bulk_g2s(dst + ST::kVR, s.vrn + tb, rows * 4, bar);
    }
    bulk_g2s(dst + ST::kVN, s.vn + tb, rows * 4, bar);
}

template <int KB, bool KP, int VB, bool VP>
__device__ __forceinline__ void produce_stage(uint32_t dst, const Slab& s, int tb, int valid, int lane) {
    using ST = Stage<KB, KP, VB, VP>;
    constexpr int R = ST::R;
    if constexpr (KB > 0) copy_rows16<ST::kRK, R>(dst + ST::kKC, s.kc + (size_t)tb * ST::kRK, valid, lane);
    if constexpr (KP) {
        copy_rows16<16, R>(dst + ST::kKS, s.ks + (size_t)tb * 16, valid, lane);
        copy_norms<R>(dst + ST::kKR, s.krn + tb, s.a16, valid, lane);
    }
    copy_norms<R>(dst + ST::kKN, s.kn + tb, s.a16, valid, lane);
    if constexpr (VB > 0) copy_rows16<ST::kRV, R>(dst + ST::kVC, s.vc + (size_t)tb * ST::kRV, valid, lane);
    if constexpr (VP) {
        copy_rows16<16, R>(dst + ST::kVS, s.vs + (size_t)tb * 16, valid, lane);
        copy_norms<R>(dst + ST::kVR, s.vrn + tb, s.a16, valid, lane);
    }
    copy_norms<R>(dst + ST::kVN, s.vn + tb, s.a16, valid, lane);
}

template <int NW>
__device__ __forceinline__ void read_words(uint32_t* w, const unsigned char* p) {
    if constexpr (NW == 1) {
        w[0] = *reinterpret_cast<const uint32_t*>(p);
    } else if constexpr (NW == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        w[0] = v.x;
        w[1] = v.y;
    } else if constexpr (NW == 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
    } else if constexpr (NW == 3) {
        const uint32_t* q = reinterpret_cast<const uint32_t*>(p);
        w[0] = q[0];
        w[1] = q[1];
        w[2] = q[2];
    }
}


// Consumer warps per CTA (one CTA per SM, plus one producer warp): prod values
// carry a second accumulator set and run fewer warps with more registers.
template <bool VP>
struct Warps {
    static constexpr int value = VP ? 7 : 11;
};

template <int KB, bool KP, int VB, bool VP>
struct Smem {
    static constexpr int W = Warps<VP>::value;    // consumer warps
    static constexpr int kThreads = (W + 1) * 32;  // and the producer warp
    // main phase: decode tables, queries, query scales, staging rings
    // tables (power-of-two sizes) largest first from a 32 KB-aligned base, so that
    // each one starts at a multiple of its own size
    static constexpr size_t kSzK = Table<KB>::kBytes, kSzV = Table<VB>::kBytes;
    static constexpr size_t kSzS = KP ? KSignTable::kBytes : 0;
    static constexpr size_t kBig = 32768;
    static constexpr size_t table_offset(int which) {  // 0 = keys, 1 = values, 2 = key signs
        const size_t sz[3] = {kSzK, kSzV, kSzS};
        size_t off = 0;
        for (int i = 0; i < 3; ++i)
            if (sz[i] == kBig) {
                if (i == which) return off;
                off += kBig;
            }
        for (int i = 0; i < 3; ++i)
            if (sz[i] != 0 && sz[i] != kBig) {
                if (i == which) return off;
                off += sz[i];
            }
        return off;
    }
    static constexpr size_t kTabK = table_offset(0), kTabV = table_offset(1), kTabS = table_offset(2);
    static constexpr size_t kQ = kSzK + kSzV + kSzS;
    static constexpr size_t kQsc = kQ + 2 * kHeads * kQRow * 4;
    static constexpr size_t kQin = kQsc + 2 * kHeads * 4;  // [kHeads][D] raw queries
    static constexpr size_t kStage = (kQin + (size_t)kHeads * D * 4 + 127) & ~(size_t)127;
    static constexpr size_t kAlignSlack = kBig - 16;  // the 32 KB-aligned base lies at most this far in
    static constexpr size_t kLimit = 232448 - 2048;   // per-CTA limit less static and reserved bytes
    static constexpr int kStagesFit = (int)((kLimit - kAlignSlack - kStage) / Stage<KB, KP, VB, VP>::kBytes);
    static constexpr int kStages = kStagesFit < kMaxStages ? kStagesFit : kMaxStages;
    static_assert(kStages >= 4, "too few staging stages fit in shared memory");
    static constexpr size_t kMain = kStage + (size_t)kStages * Stage<KB, KP, VB, VP>::kBytes;
    // combine phase (reuses the same bytes): per-warp maxima, sums, weights and
    // accumulators (the latter in fragment order: [warp][m][i][lane])
    static constexpr size_t kWM = 0;
    static constexpr size_t kWL = kWM + W * kHeads * 4;
    static constexpr size_t kWF = kWL + W * kHeads * 4;
    static constexpr size_t kWO = kWF + W * kHeads * 4;
    static constexpr size_t kWO2 = kWO + (size_t)W * kHeads * D * 4;
    static constexpr size_t kCombine = kWO2 + (VP ? (size_t)W * kHeads * D * 4 : 0);
    // merge phase of the last CTA of a group (reuses the same bytes again)
    static constexpr int kMaxSplits = kMaxSplitsMerged;
    static constexpr size_t kMW = 0;                                      // [kHeads][kMaxSplits] weights
    static constexpr size_t kML = kMW + (size_t)kHeads * kMaxSplits * 4;  // [kHeads] 1/l
    static constexpr int kMRow = D + 8;                                   // padded row: 2-way LDS.64 conflicts
    static constexpr size_t kMO = (kML + kHeads * 4 + 15) & ~(size_t)15;  // [2][kHeads][kMRow] merged acc
    static constexpr int kMC = VP ? 16 : 32;                              // splits staged per round
    static constexpr size_t kMS = kMO + 2 * (size_t)kHeads * kMRow * 4;   // [VP ? 2 : 1][kHeads][kMC][D] partials
    static constexpr size_t kMerge = kMS + (VP ? 2 : 1) * (size_t)kMC * kHeads * D * 4;
    static_assert(kQin % 16 == 0 && kMS % 16 == 0, "cp.async destinations must be 16-byte aligned");
    static constexpr size_t kBytes0 = kMain + kAlignSlack > kCombine ? kMain + kAlignSlack : kCombine;
    static constexpr size_t kBytes = kBytes0 > kMerge ? kBytes0 : kMerge;
};

// Per-lane running state of the online softmax (head g of the lane; the four
// lanes of a quad share it) and the value accumulators (heads 2c, 2c + 1).
template <bool VP>
struct Acc {
    float O[kMT][4];
    float O2[VP ? kMT : 1][4];
    float M, Mt, l;
};

// One 16-token step of a warp: tokens tb … tb + 15 (FULL: all below t1), rows
// r0 … r0 + 15 of the stage at stp.  AQ[kb] = [Q′_hi; Q′_lo] fragments of head g,
// AS[kb] = [Q″_hi; Q″_lo].  Lane (g, c) ends with the weights of head g for tokens 2c, 2c + 1 and
// 8 + 2c, 9 + 2c, which are the B fragment of the value MMA.
template <int KB, bool KP, int VB, bool VP, bool FULL>
__device__ __forceinline__ void step(Acc<VP>& st, const unsigned char* stp, int r0, int tb, int t1,
                                     const KDecoder<KB>& dk, const Decoder<VB>& dv, const SignDecoder& ds,
                                     uint32_t stab, const uint32_t (&AQ)[kKB][4], const uint32_t (&AS)[kKB][4],
                                     float fK, float fS, const SplitArgs& a, size_t head0, int G, int g, int c) {
    using ST = Stage<KB, KP, VB, VP>;
    // ---- scores of head g: S1 = [Q′_hi; Q′_lo]·K̃ᵀ (codes), S2 = [Q″_hi; Q″_lo]·Zᵀ (QJL signs)
    // accumulator of group n: [0] (hi, token 2c) [1] (hi, 2c + 1) [2] (lo, 2c) [3] (lo, 2c + 1)
    // Each score sums its k16 blocks in two independent accumulator chains (even
    // and odd blocks), so that an MMA need not wait for the one before it.
    float S1[2][4], S2[2][4], S1x[2][4], S2x[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
#pragma unroll
        for (int i = 0; i < 4; ++i) S1[n][i] = S2[n][i] = S1x[n][i] = S2x[n][i] = 0.f;
        if constexpr (KB > 0) {
            uint32_t w[KB];
            read_words<KB>(w, stp + ST::kKC + (r0 + 8 * n + g) * ST::kRK + c * (KB * 4));
#pragma unroll
            for (int kb = 0; kb < kKB; ++kb) {
                uint32_t b0, b1;
                dk.frag(w, kb, b0, b1);
                mma16816((kb & 1) ? S1x[n] : S1[n], AQ[kb][0], AQ[kb][1], AQ[kb][2], AQ[kb][3], b0, b1);
            }
        }
        if constexpr (KP) {
            const uint32_t ws = *reinterpret_cast<const uint32_t*>(stp + ST::kKS + (r0 + 8 * n + g) * 16 + c * 4);
#pragma unroll
            for (int j = 0; j < kKB / 2; ++j) {
                const uint4 f = lds128(field_off<8, 7>(&ws, 8 * j) | stab);
                mma16816(S2[n], AS[2 * j][0], AS[2 * j][1], AS[2 * j][2], AS[2 * j][3], f.x, f.y);
                mma16816(S2x[n], AS[2 * j + 1][0], AS[2 * j + 1][1], AS[2 * j + 1][2], AS[2 * j + 1][3], f.z, f.w);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            S1[n][i] += S1x[n][i];
            S2[n][i] += S2x[n][i];
        }
    }
    // this lane's tokens: i = 0, 1 → 2c, 2c + 1; i = 2, 3 → 8 + 2c, 9 + 2c
    auto norms = [&](int off, float (&v)[4]) {
        const float2 x = *reinterpret_cast<const float2*>(stp + off + 4 * r0 + 8 * c);
        const float2 y = *reinterpret_cast<const float2*>(stp + off + 4 * r0 + 32 + 8 * c);
        v[0] = x.x;
        v[1] = x.y;
        v[2] = y.x;
        v[3] = y.y;
    };
    float kn[4], vn[4], kr[4];
    norms(ST::kKN, kn);
    norms(ST::kVN, vn);
    if constexpr (KP) norms(ST::kKR, kr);
    // z = s·log2e + log2‖v‖ (the exponent of the value weight), −∞ past the chunk
    float z[4], lv[4], rv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int n = i >> 1, j = i & 1;
        const float vv = fmaxf(vn[i], 1e-30f);
        lv[i] = lg2(vv);
        rv[i] = rcp(vv);
        float v = fK * (S1[n][j] + S1[n][2 + j]);
        if constexpr (KP) v = fmaf(fS * kr[i], S2[n][j] + S2[n][2 + j], v);
        z[i] = fmaf(kn[i], v, lv[i]);
        if constexpr (!FULL)
            if (tb + 8 * n + 2 * c + j >= t1) z[i] = -INFINITY;
    }
    if (a.scores != nullptr && g < G) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = tb + 8 * (i >> 1) + 2 * c + (i & 1);
            if (FULL || t < t1) a.scores[(head0 + g) * a.T_max + t] = (z[i] - lv[i]) * kLn2;
        }
    }

    // ---- online softmax with a lazily raised maximum (head g, shared by the quad)
    const float zm = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
    if (__any_sync(0xffffffffu, zm > st.Mt)) {
        float mx = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float Mn = fmaxf(st.M, mx);
        const float corr = Mn == -INFINITY ? 1.f : ex2(st.M - Mn);  // 0 on the first raise (M = −∞)
        st.M = Mn;
        st.Mt = Mn + kSlack;
        st.l *= corr;
        // the accumulators hold heads 2c and 2c + 1, whose state lives in quads 2c, 2c + 1
        const float cA = __shfl_sync(0xffffffffu, corr, 8 * c), cB = __shfl_sync(0xffffffffu, corr, 8 * c + 4);
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
            st.O[m][0] *= cA;
            st.O[m][1] *= cB;
            st.O[m][2] *= cA;
            st.O[m][3] *= cB;
            if constexpr (VP) {
                st.O2[m][0] *= cA;
                st.O2[m][1] *= cB;
                st.O2[m][2] *= cA;
                st.O2[m][3] *= cB;
            }
        }
    }
    float pv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        pv[i] = ex2(z[i] - st.M);
        st.l = fmaf(pv[i], rv[i], st.l);
    }
    // B fragment of the value MMA: head g, tokens (2c, 2c + 1) and (8 + 2c, 9 + 2c)
    const uint32_t PB0 = pack_h2(pv[0], pv[1]);
    const uint32_t PB1 = pack_h2(pv[2], pv[3]);

    // ---- values: Oᵀ += Ṽᵀ·P′ᵀ in the rotated frame
    if constexpr (VB > 0) {
        uint32_t vwA[VB], vwB[VB];
        read_words<VB>(vwA, stp + ST::kVC + (r0 + g) * ST::kRV + c * (VB * 4));
        read_words<VB>(vwB, stp + ST::kVC + (r0 + g + 8) * ST::kRV + c * (VB * 4));
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
            uint32_t x0, x1, y0, y1;
            dv.pairs(vwA, m, x0, x1);
            dv.pairs(vwB, m, y0, y1);
            mma16816(st.O[m], mov_trans(x0), mov_trans(x1), mov_trans(y0), mov_trans(y1), PB0, PB1);
        }
    }
    if constexpr (VP) {
        float vr[4];
        norms(ST::kVR, vr);
        if constexpr (!FULL) {
            // rows past the chunk may hold anything (bulk staging copies whole tiles)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (tb + 8 * (i >> 1) + 2 * c + (i & 1) >= t1) vr[i] = 0.f;
        }
        const uint32_t QB0 = pack_h2(pv[0] * a.vgamma * vr[0], pv[1] * a.vgamma * vr[1]);
        const uint32_t QB1 = pack_h2(pv[2] * a.vgamma * vr[2], pv[3] * a.vgamma * vr[3]);
        const uint32_t vsA = *reinterpret_cast<const uint32_t*>(stp + ST::kVS + (r0 + g) * 16 + c * 4);
        const uint32_t vsB = *reinterpret_cast<const uint32_t*>(stp + ST::kVS + (r0 + g + 8) * 16 + c * 4);
#pragma unroll
        for (int m = 0; m < kMT / 2; ++m) {
            uint32_t pa[4], pb[4];
            ds.quad(vsA, m, pa);
            ds.quad(vsB, m, pb);
            mma16816(st.O2[2 * m], mov_trans(pa[0]), mov_trans(pa[1]), mov_trans(pb[0]), mov_trans(pb[1]), QB0, QB1);
            mma16816(st.O2[2 * m + 1], mov_trans(pa[2]), mov_trans(pa[3]), mov_trans(pb[2]), mov_trans(pb[3]), QB0,
                     QB1);
        }
    }
}

// The step for at most four query heads per KV head (G4).  With [Q′_hi; Q′_lo] as
// the A operand, four heads would fill only half of the MMA's 16 rows; here the
// keys (and the QJL signs) are the A operand instead, 16 tokens × 16 dims, and
// the queries the B operand, 8 columns (head h: Q′_hi in column 2h, Q′_lo in
// 2h + 1), so each k16 block is one MMA for the whole tile instead of two.  Lane
// (g, c) ends with head c's scores of tokens g and g + 8 (the two columns of head
// c are the lane's accumulator pair).  The softmax weights are gathered into the
// token × head tile that movmatrix transposes into the B fragment of the value
// MMA, which is unchanged.  BQ[kb], BS[kb]: this lane's B fragments (column g).
template <int KB, bool KP, int VB, bool VP, bool FULL>
__device__ __forceinline__ void step4(Acc<VP>& st, const unsigned char* stp, int r0, int tb, int t1,
                                      const KDecoder<KB>& dk, const Decoder<VB>& dv, const SignDecoder& ds,
                                      uint32_t stab, const uint32_t (&BQ)[kKB][2], const uint32_t (&BS)[kKB][2],
                                      float fK, float fS, const SplitArgs& a, size_t head0, int G, int g, int c) {
    using ST = Stage<KB, KP, VB, VP>;
    // accumulators: [0] token g column 2c (hi), [1] token g column 2c + 1 (lo),
    // [2], [3] the same for token g + 8; even and odd k16 blocks in two chains
    float S1[4] = {0.f, 0.f, 0.f, 0.f}, S1x[4] = {0.f, 0.f, 0.f, 0.f};
    float S2[4] = {0.f, 0.f, 0.f, 0.f}, S2x[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (KB > 0) {
        uint32_t w0[KB], w1[KB];
        read_words<KB>(w0, stp + ST::kKC + (r0 + g) * ST::kRK + c * (KB * 4));
        read_words<KB>(w1, stp + ST::kKC + (r0 + 8 + g) * ST::kRK + c * (KB * 4));
#pragma unroll
        for (int kb = 0; kb < kKB; ++kb) {
            // a token's B fragment of the other orientation is its row of the A fragment
            uint32_t a0, a1, a2, a3;
            dk.frag(w0, kb, a0, a2);
            dk.frag(w1, kb, a1, a3);
            mma16816((kb & 1) ? S1x : S1, a0, a1, a2, a3, BQ[kb][0], BQ[kb][1]);
        }
    }
    if constexpr (KP) {
        const uint32_t ws0 = *reinterpret_cast<const uint32_t*>(stp + ST::kKS + (r0 + g) * 16 + c * 4);
        const uint32_t ws1 = *reinterpret_cast<const uint32_t*>(stp + ST::kKS + (r0 + 8 + g) * 16 + c * 4);
#pragma unroll
        for (int j = 0; j < kKB / 2; ++j) {
            const uint4 f0 = lds128(field_off<8, 7>(&ws0, 8 * j) | stab);
            const uint4 f1 = lds128(field_off<8, 7>(&ws1, 8 * j) | stab);
            mma16816(S2, f0.x, f1.x, f0.y, f1.y, BS[2 * j][0], BS[2 * j][1]);
            mma16816(S2x, f0.z, f1.z, f0.w, f1.w, BS[2 * j + 1][0], BS[2 * j + 1][1]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        S1[i] += S1x[i];
        S2[i] += S2x[i];
    }
    // this lane's tokens: i = 0 → g, i = 1 → g + 8
    auto norm2 = [&](int off, float (&v)[2]) {
        v[0] = *reinterpret_cast<const float*>(stp + off + 4 * (r0 + g));
        v[1] = *reinterpret_cast<const float*>(stp + off + 4 * (r0 + 8 + g));
    };
    float kn[2], vn[2], kr[2];
    norm2(ST::kKN, kn);
    norm2(ST::kVN, vn);
    if constexpr (KP) norm2(ST::kKR, kr);
    float z[2], lv[2], rv[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float vv = fmaxf(vn[i], 1e-30f);
        lv[i] = lg2(vv);
        rv[i] = rcp(vv);
        float v = fK * (S1[2 * i] + S1[2 * i + 1]);
        if constexpr (KP) v = fmaf(fS * kr[i], S2[2 * i] + S2[2 * i + 1], v);
        z[i] = fmaf(kn[i], v, lv[i]);
        if constexpr (!FULL)
            if (tb + g + 8 * i >= t1) z[i] = -INFINITY;
    }
    if (a.scores != nullptr && c < G) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int t = tb + g + 8 * i;
            if (FULL || t < t1) a.scores[(head0 + c) * a.T_max + t] = (z[i] - lv[i]) * kLn2;
        }
    }

    // ---- online softmax of head c (shared by the eight lanes with this c)
    const float zm = fmaxf(z[0], z[1]);
    if (__any_sync(0xffffffffu, zm > st.Mt)) {
        float mx = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float Mn = fmaxf(st.M, mx);
        const float corr = Mn == -INFINITY ? 1.f : ex2(st.M - Mn);  // 0 on the first raise (M = −∞)
        st.M = Mn;
        st.Mt = Mn + kSlack;
        st.l *= corr;
        // the value accumulators hold heads 2c and 2c + 1 (lanes 2c and 2c + 1 keep their
        // state); for c ≥ 2 they hold no head and stay zero
        const float cA = __shfl_sync(0xffffffffu, corr, 2 * c), cB = __shfl_sync(0xffffffffu, corr, 2 * c + 1);
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
            st.O[m][0] *= cA;
            st.O[m][1] *= cB;
            st.O[m][2] *= cA;
            st.O[m][3] *= cB;
            if constexpr (VP) {
                st.O2[m][0] *= cA;
                st.O2[m][1] *= cB;
                st.O2[m][2] *= cA;
                st.O2[m][3] *= cB;
            }
        }
    }
    float pv[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        pv[i] = ex2(z[i] - st.M);
        st.l = fmaf(pv[i], rv[i], st.l);
    }
    // token × head tile X (block 0: tokens 0–7, block 1: 8–15): lane (g, c) holds
    // X[g][2c], X[g][2c + 1], the weights of heads 2c and 2c + 1 for token g (lanes
    // (g, 2c) and (g, 2c + 1)), zero for c ≥ 2; its transpose gives lane (g, c) head
    // g's weights of tokens 2c, 2c + 1 — the value MMA's B fragment
    const int srcA = 4 * g + ((2 * c) & 3), srcB = 4 * g + ((2 * c + 1) & 3);
    auto to_b = [&](float x) -> uint32_t {
        const float xa = __shfl_sync(0xffffffffu, x, srcA), xb = __shfl_sync(0xffffffffu, x, srcB);
        return mov_trans(c < 2 ? pack_h2(xa, xb) : 0u);
    };
    const uint32_t PB0 = to_b(pv[0]);
    const uint32_t PB1 = to_b(pv[1]);

    // ---- values: Oᵀ += Ṽᵀ·P′ᵀ in the rotated frame (as in step)
    if constexpr (VB > 0) {
        uint32_t vwA[VB], vwB[VB];
        read_words<VB>(vwA, stp + ST::kVC + (r0 + g) * ST::kRV + c * (VB * 4));
        read_words<VB>(vwB, stp + ST::kVC + (r0 + g + 8) * ST::kRV + c * (VB * 4));
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
            uint32_t x0, x1, y0, y1;
            dv.pairs(vwA, m, x0, x1);
            dv.pairs(vwB, m, y0, y1);
            mma16816(st.O[m], mov_trans(x0), mov_trans(x1), mov_trans(y0), mov_trans(y1), PB0, PB1);
        }
    }
    if constexpr (VP) {
        float vr[2];
        norm2(ST::kVR, vr);
        if constexpr (!FULL) {
            // rows past the chunk may hold anything (bulk staging copies whole tiles)
#pragma unroll
            for (int i = 0; i < 2; ++i)
                if (tb + g + 8 * i >= t1) vr[i] = 0.f;
        }
        const uint32_t QB0 = to_b(pv[0] * a.vgamma * vr[0]);
        const uint32_t QB1 = to_b(pv[1] * a.vgamma * vr[1]);
        const uint32_t vsA = *reinterpret_cast<const uint32_t*>(stp + ST::kVS + (r0 + g) * 16 + c * 4);
        const uint32_t vsB = *reinterpret_cast<const uint32_t*>(stp + ST::kVS + (r0 + g + 8) * 16 + c * 4);
#pragma unroll
        for (int m = 0; m < kMT / 2; ++m) {
            uint32_t pa[4], pb[4];
            ds.quad(vsA, m, pa);
            ds.quad(vsB, m, pb);
            mma16816(st.O2[2 * m], mov_trans(pa[0]), mov_trans(pa[1]), mov_trans(pb[0]), mov_trans(pb[1]), QB0, QB1);
            mma16816(st.O2[2 * m + 1], mov_trans(pa[2]), mov_trans(pa[3]), mov_trans(pb[2]), mov_trans(pb[3]), QB0,
                     QB1);
        }
    }
}

// Last CTA of a (batch, KV head, head block) group: combine the n_splits
// partials of its G heads and write out = Π_vᵀ·acc/l (+ S_vᵀ·acc2/l).
template <int KB, bool KP, int VB, bool VP>
__device__ __forceinline__ void merge_group(const SplitArgs& a, unsigned char* smem, size_t head0, int G) {
    using SM = Smem<KB, KP, VB, VP>;
    constexpr int NT = SM::kThreads, NW = NT / 32, MR = SM::kMRow;
    float* wts = reinterpret_cast<float*>(smem + SM::kMW);   // [kHeads][kMaxSplits]
    float* linv = reinterpret_cast<float*>(smem + SM::kML);  // [kHeads]
    float* mo = reinterpret_cast<float*>(smem + SM::kMO);    // [2][kHeads][MR]: acc/l, acc2/l
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int ns = a.n_splits;
    // out = Π_vᵀ·(acc/l) (+ S_vᵀ·(acc2/l)) on the tensor cores: warp w takes the 8
    // output dims 8·job for job = w, w + NW, …; with mse values its Π_vᵀ operand is
    // loaded now, so that the load overlaps the split sums
    constexpr int kJobs = D / 8, kPer = (kJobs + NW - 1) / NW;
    constexpr bool kEarly = !VP;  // prod values: two matrices, loaded per job (registers)
    uint4 bh[kEarly ? kPer : 1][kKB / 2], bl[kEarly ? kPer : 1][kKB / 2];
    if constexpr (kEarly) {
#pragma unroll
        for (int u = 0; u < kPer; ++u)
            if (warp + u * NW < kJobs) hilo_b(a.vPiT_hi, a.vPiT_lo, 8 * (warp + u * NW), g, c, bh[u], bl[u]);
    }
    // the split partials, kMC splits per round, brought into shared memory by one
    // bulk copy per head (a head's splits are contiguous rows) while the split
    // weights are formed
    __shared__ __align__(8) uint64_t s_mbar;
    float* stg = reinterpret_cast<float*>(smem + SM::kMS);
    constexpr int kMC = SM::kMC;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&s_mbar, 1);
        sm100::fence_barrier_init();
    }
    __syncthreads();
    auto stage_round = [&](int s0) {  // thread 0; the previous contents have been read
        if (threadIdx.x == 0) {
            const uint32_t bytes = (uint32_t)min(kMC, ns - s0) * D * 4;
            asm volatile("fence.proxy.async;" ::: "memory");
            sm100::mbar_arrive_expect_tx(&s_mbar, (VP ? 2 : 1) * G * bytes);
#pragma unroll
            for (int mtx = 0; mtx < (VP ? 2 : 1); ++mtx)
                for (int h = 0; h < G; ++h)
                    bulk_g2s(smem_addr(stg + (size_t)(mtx * kHeads + h) * kMC * D),
                             (mtx ? a.pacc2 : a.pacc) + ((head0 + h) * ns + s0) * D, bytes, smem_addr(&s_mbar));
        }
    };
    stage_round(0);
    if (warp < G) {
        // split weights of head `warp`: every pm and pl load of the head in flight at once
        constexpr int kR = SM::kMaxSplits / 32;
        const size_t hs = (head0 + warp) * ns;
        float pmv[kR], plv[kR];
#pragma unroll
        for (int k = 0; k < kR; ++k) {
            const int sp = lane + 32 * k;
            pmv[k] = sp < ns ? __ldcg(a.pm + hs + sp) : -INFINITY;
            plv[k] = sp < ns ? __ldcg(a.pl + hs + sp) : 0.f;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < kR; ++k) mx = fmaxf(mx, pmv[k]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float l = 0.f;
#pragma unroll
        for (int k = 0; k < kR; ++k) {
            const int sp = lane + 32 * k;
            if (sp < ns) {
                const float f = mx == -INFINITY ? 0.f : ex2((pmv[k] - mx) * kLog2e);
                wts[warp * SM::kMaxSplits + sp] = f;
                l = fmaf(f, plv[k], l);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) linv[warp] = l > 0.f ? 1.f / l : 0.f;
    }
    // Σ over splits from shared memory: thread t < kHeads·D/4 sums four dims of one head
    const int th = threadIdx.x / (D / 4), tj = threadIdx.x % (D / 4);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f), o2 = o;
    for (int s0 = 0, round = 0; s0 < ns; s0 += kMC, ++round) {
        const bool ok = sm100::mbar_wait(&s_mbar, (uint32_t)(round & 1), a.status, kDecodeMergeTimeout);
        __syncthreads();  // this round's partials (and, first time, the weights) are visible
        const int nsc = min(kMC, ns - s0);
        if (ok && th < G) {
            const float* w = wts + th * SM::kMaxSplits + s0;
            const float4* x = reinterpret_cast<const float4*>(stg) + (size_t)th * kMC * (D / 4) + tj;
            const float4* x2 = x + (size_t)kHeads * kMC * (D / 4);
            for (int sp = 0; sp < nsc; ++sp) {
                const float ws = w[sp];
                const float4 v = x[sp * (D / 4)];
                o = make_float4(fmaf(ws, v.x, o.x), fmaf(ws, v.y, o.y), fmaf(ws, v.z, o.z), fmaf(ws, v.w, o.w));
                if constexpr (VP) {
                    const float4 v2 = x2[sp * (D / 4)];
                    o2 = make_float4(fmaf(ws, v2.x, o2.x), fmaf(ws, v2.y, o2.y), fmaf(ws, v2.z, o2.z),
                                     fmaf(ws, v2.w, o2.w));
                }
            }
        }
        if (s0 + kMC < ns) {
            __syncthreads();  // the staged round has been read
            stage_round(s0 + kMC);
        }
    }
    if (th < kHeads) {  // heads past G: zero
        const float li = th < G ? linv[th] : 0.f;
        *reinterpret_cast<float4*>(mo + th * MR + 4 * tj) = make_float4(o.x * li, o.y * li, o.z * li, o.w * li);
        if constexpr (VP)
            *reinterpret_cast<float4*>(mo + kHeads * MR + th * MR + 4 * tj) =
                make_float4(o2.x * li, o2.y * li, o2.z * li, o2.w * li);
    }
    __syncthreads();
    uint32_t A[kKB][4], A2[VP ? kKB : 1][4];
    hilo_a(mo + g * MR, c, A);
    if constexpr (VP) hilo_a(mo + kHeads * MR + g * MR, c, A2);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int job = warp + u * NW;
        if (job >= kJobs) break;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (kEarly) {
            hilo_mma(acc, A, bh[u], bl[u]);
        } else {
            uint4 ph[kKB / 2], pl[kKB / 2], sh[kKB / 2], sl[kKB / 2];
            hilo_b(a.vPiT_hi, a.vPiT_lo, 8 * job, g, c, ph, pl);
            hilo_b(a.vST_hi, a.vST_lo, 8 * job, g, c, sh, sl);
            hilo_mma(acc, A, ph, pl);
            hilo_mma(acc, A2, sh, sl);
        }
        if (g < G)
            *reinterpret_cast<float2*>(a.out + (head0 + g) * D + 8 * job + 2 * c) =
                make_float2(acc[0] + acc[2], acc[1] + acc[3]);
    }
}

// AA: launched behind the decode-step append (a.after_append), which writes no
// cache row below the length it starts from: the stages wholly below that
// length are streamed and consumed before griddepcontrol.wait.
// G4: at most four query heads per KV head, stepped by step4.
template <int KB, bool KP, int VB, bool VP, bool AA, bool G4>
__global__ void __launch_bounds__((Warps<VP>::value + 1) * 32, 1) decode_split_mma_kernel(const SplitArgs a) {
    using SM = Smem<KB, KP, VB, VP>;
    using ST = Stage<KB, KP, VB, VP>;
    constexpr int W = SM::W;
    extern __shared__ __align__(128) unsigned char smem[];
    // main-phase regions start at the first 32 KB-aligned shared address
    const uint32_t sbase = smem_addr(smem);
    unsigned char* mp = smem + (((sbase + (uint32_t)SM::kBig - 1u) & ~((uint32_t)SM::kBig - 1u)) - sbase);
    float* qsh = reinterpret_cast<float*>(mp + SM::kQ);     // [2][kHeads][kQRow]: q′, q″ (see qidx)
    float* qsc = reinterpret_cast<float*>(mp + SM::kQsc);   // [2][kHeads]
    __shared__ int s_last;

    const int hb = blockIdx.y % a.n_hblocks, kvh = blockIdx.y / a.n_hblocks;
    const int G = min(kHeads, a.G - hb * kHeads);
    // the grid is (batch, KV head × head block, split): CTAs start split by split,
    // so with ragged lengths the full chunks go first and the partial and empty
    // ones (the later splits of short sequences) last
    const int split = blockIdx.z, b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int t0 = split * a.chunk;
    // Lengths, cache planes, merge tickets and (unless a.after_append) the queries may
    // come from the kernels launched before this one, whose tails this grid may
    // overlap as a programmatic dependent: each branch reads them only after
    // griddepcontrol.wait, which returns at once for an ordinary launch.
    int t1 = t0, ntiles = 0, nstages = 0;
    auto read_length = [&]() {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int L = a.seq_lens[b];
        L = L < 0 ? 0 : (L > a.T_max ? a.T_max : L);
        t1 = min(t0 + a.chunk, L);
        ntiles = t1 > t0 ? (t1 - t0 + kTile - 1) / kTile : 0;
        nstages = (ntiles + ST::R / kTile - 1) / (ST::R / kTile);
    };
    const size_t head0 = (size_t)b * a.Hq + (size_t)kvh * a.G + (size_t)hb * kHeads;
    const int64_t rowbase = ((int64_t)b * a.Hkv + kvh) * a.T_max;

    // the bf16 hi/lo matrices every CTA reads (Π_k, S_k for the query rotation) or
    // the merging CTAs read (Π_vᵀ, S_vᵀ): one L2 prefetch per 128-byte line, spread
    // over the CTAs of the grid, kept with the evict-last priority
    {
        const int nct = gridDim.x * gridDim.y * gridDim.z;
        const int cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        constexpr int kLines = D * D * 2 / 128;  // lines of one bf16 matrix
        constexpr int kMats = 4 + (KP ? 2 : 0) + (VP ? 2 : 0);
        const int l = cta + nct * (int)threadIdx.x;
        if (l < kMats * kLines) {
            int m = l / kLines;
            if (!KP && m >= 4) m += 2;  // skip S_k
            const uint16_t* base = m == 0 ? a.kPi_hi : m == 1 ? a.kPi_lo : m == 2 ? a.vPiT_hi : m == 3 ? a.vPiT_lo
                                 : m == 4 ? a.kS_hi : m == 5 ? a.kS_lo : m == 6 ? a.vST_hi : a.vST_lo;
            asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(base + 64 * (l % kLines)));
        }
    }

    Slab sl;
    sl.a16 = (rowbase & 3) == 0;
    sl.kc = a.kcodes + (size_t)rowbase * (KB * 16);
    sl.ks = a.ksigns + (size_t)rowbase * 16;
    sl.kn = a.knorm + rowbase;
    sl.krn = a.krnorm + rowbase;
    sl.vc = a.vcodes + (size_t)rowbase * (VB * 16);
    sl.vs = a.vsigns + (size_t)rowbase * 16;
    sl.vn = a.vnorm + rowbase;
    sl.vrn = a.vrnorm + rowbase;

    // ---- staging ring: warp W produces, warps 0 … W − 1 consume 16-token tiles
    const uint32_t ring = smem_addr(mp + SM::kStage);
    __shared__ __align__(8) uint64_t s_full[SM::kStages], s_empty[SM::kStages];
    const bool producer = warp == W;
    // bulk staging when every slab's norm rows start on a 16-byte boundary:
    // one lane, one copy per plane and stage
    const bool bulk = (a.T_max & 3) == 0;
    // AA: stages of this chunk wholly below L_pre − 1 (L_pre: the length read
    // before the wait, the append's starting length or that plus one, so every
    // row below L_pre − 1 was complete before the append started)
    int ns_safe = 0;
    if constexpr (AA) {
        if (bulk) {
            int Lp;
            asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(Lp) : "l"(a.seq_lens + b) : "memory");
            Lp = Lp > a.T_max ? a.T_max : Lp;
            const int safe = min(t0 + a.chunk, Lp - 1) - t0;
            ns_safe = safe > 0 ? safe / ST::R : 0;
        }
    }
    auto produce = [&](int i) {
        const int tb = t0 + i * ST::R;
        const uint32_t dst = ring + (uint32_t)((i % SM::kStages) * ST::kBytes);
        const uint32_t bar = smem_addr(&s_full[i % SM::kStages]);
        if (bulk) {
            if (lane == 0) produce_stage_bulk<KB, KP, VB, VP>(dst, bar, sl, tb, a.T_max);
        } else {
            produce_stage<KB, KP, VB, VP>(dst, sl, tb, t1 - tb, lane);
            // the stage's full barrier counts one arrival per producer lane, made when
            // that lane's copies have landed
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
        }
    };
    // the stage barriers exist before anyone waits on them; from here on the
    // producer streams stages and the consumers prepare tables and queries
    // without waiting for it (their barriers are named barrier 1, W warps)
    if (producer && lane == 0) {
        for (int i = 0; i < SM::kStages; ++i) {
            sm100::mbar_init(&s_full[i], bulk ? 1 : 32);
            sm100::mbar_init(&s_empty[i], ST::R / kTile);
        }
        sm100::fence_barrier_init();
    }
    // A CTA whose chunk starts at or past its sequence's length has no tokens: it
    // skips the staging and the prologue and contributes an empty partial (M = −∞,
    // l = 0) to the merge.  Thread 0 reads the length before griddepcontrol.wait as
    // a hint and, when it says "empty", waits and reads it again before deciding
    // for the CTA (a chunk that the hint wrongly calls empty takes the ordinary
    // path, only without its prologue overlap); the ragged batched workload has
    // about one such CTA per sequence in four.  Only the small-group variant (G4,
    // the batched workload's) has this path: in the eight-head variant the extra
    // branch changed the register allocation and cost 3 % of the 131072-token
    // decode.  Behind the decode-step append the length read after the wait is
    // the bumped one, so a chunk that starts at the new row is not skipped.
    constexpr bool kSkip = G4;
    __shared__ int s_skip;
    if constexpr (kSkip) {
        if (threadIdx.x == 0) {
            int Lh;
            asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(Lh) : "l"(a.seq_lens + b) : "memory");
            int skip = 0;
            if (t0 >= Lh) {
                asm volatile("griddepcontrol.wait;" ::: "memory");
                const int L = a.seq_lens[b];
                skip = t0 >= L;
            }
            s_skip = skip;
        }
    }
    __syncthreads();
    const bool skip = kSkip && s_skip != 0;
    auto consumers_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(W * 32) : "memory"); };

    Acc<VP> st;
#pragma unroll
    for (int m = 0; m < kMT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            st.O[m][i] = 0.f;
            if constexpr (VP) st.O2[m][i] = 0.f;
        }
    st.M = -INFINITY;
    st.Mt = -INFINITY;
    st.l = 0.f;

    if (skip) {
        // no tokens: straight to the combine (the partial is M = −∞, l = 0, O = 0)
    } else if (producer) {
        // ---- producer: the first stages, then each stage again once its four
        // tiles have been consumed
        bool live = true;
        if constexpr (AA) {  // the stages below ns_safe before the wait
            for (int i = 0; i < ns_safe; ++i) {
                if (i >= SM::kStages) {
                    live = __all_sync(0xffffffffu, sm100::mbar_wait(&s_empty[i % SM::kStages],
                                                                    (uint32_t)((i / SM::kStages - 1) & 1), a.status,
                                                                    kDecodeStageTimeout));
                    if (!live) break;
                }
                produce(i);
            }
        }
        read_length();
        if (live) {
            for (int i = ns_safe; i < min(nstages, SM::kStages); ++i) produce(i);
            for (int i = max(SM::kStages, ns_safe); i < nstages; ++i) {
                const bool ok = sm100::mbar_wait(&s_empty[i % SM::kStages], (uint32_t)((i / SM::kStages - 1) & 1),
                                                 a.status, kDecodeStageTimeout);
                if (!__all_sync(0xffffffffu, ok)) break;
                produce(i);
            }
        }
        cp_async_wait<0>();  // every copy this warp issued has landed
    } else {
        // ---- prologue (consumer warps): decode tables, queries, query scales
        constexpr int NC = W * 32;
        // q′ = Π_k·q and q″ = S_k·q on the tensor cores (hilo_*): warp w takes the
        // 8-dim tiles w, w + W, … of the two products; the matrix loads and the raw
        // query loads are issued before the table fill so that their latency
        // overlaps it
        constexpr int kJobs = (KP ? 2 : 1) * (D / 8);
        constexpr int kPer = (kJobs + W - 1) / W;
        uint4 bh[kPer][kKB / 2], bl[kPer][kKB / 2];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int job = warp + u * W;
            if (job < kJobs) {
                const bool second = job >= D / 8;
                hilo_b(second ? a.kS_hi : a.kPi_hi, second ? a.kS_lo : a.kPi_lo, 8 * (job % (D / 8)), g, c, bh[u],
                       bl[u]);
            }
        }
        // the raw queries of this head block (rows as stored, bf16 or fp32; heads
        // past G zero) copied into shared memory: while the tables are filled when
        // they may be read early, else after the tables and griddepcontrol.wait
        unsigned char* qin = mp + SM::kQin;  // [kHeads][D] elements of the query dtype
        auto load_q = [&]() {
            const int rowq = a.q_f32 ? D / 4 : D / 8;  // 16-byte pieces per head row
            const unsigned char* qb = static_cast<const unsigned char*>(a.q) + head0 * D * (a.q_f32 ? 4 : 2);
            for (int idx = threadIdx.x; idx < kHeads * rowq; idx += NC) {
                const bool live = idx / rowq < G;
                cp_async16(smem_addr(qin) + 16u * (uint32_t)idx, live ? qb + 16 * idx : qb, live ? 16u : 0u);
            }
            cp_async_commit();
        };
        if (a.after_append) load_q();
        Table<KB>::fill(mp + SM::kTabK, a.kcb, threadIdx.x, NC);
        Table<VB>::fill(mp + SM::kTabV, a.vcb, threadIdx.x, NC);
        if constexpr (KP) KSignTable::fill(mp + SM::kTabS, threadIdx.x, NC);
        if (!a.after_append) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            load_q();
        }
        cp_async_wait<0>();
        consumers_sync();
        {
            uint32_t A[kKB][4];
            if (a.q_f32)
                hilo_a(reinterpret_cast<const float*>(qin) + g * D, c, A);
            else
                hilo_a(reinterpret_cast<const __nv_bfloat16*>(qin) + g * D, c, A);
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int job = warp + u * W;
                if (job < kJobs) {
                    const int second = job >= D / 8, j0 = 8 * (job % (D / 8));
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    hilo_mma(acc, A, bh[u], bl[u]);
                    float* o = qsh + (second ? kHeads * kQRow : 0) + qidx(g, j0 + 2 * c);
                    o[0] = acc[0] + acc[2];
                    o[1] = acc[1] + acc[3];
                }
            }
        }
        consumers_sync();
        for (int h = warp; h < kHeads; h += W) {  // W may be below kHeads (prod values)
            // max|q′| (and max|q″|) of head h
            float m1 = 0.f, m2 = 0.f;
            for (int j = lane; j < D; j += 32) {
                m1 = fmaxf(m1, fabsf(qsh[qidx(h, j)]));
                if constexpr (KP) m2 = fmaxf(m2, fabsf(qsh[kHeads * kQRow + qidx(h, j)]));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
                m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
            }
            if (lane == 0) {
                qsc[h] = m1 > 0.f ? m1 : 1.f;
                qsc[kHeads + h] = m2 > 0.f ? m2 : 1.f;
            }
        }
        consumers_sync();

        if constexpr (!AA) read_length();
        // A fragments of head hq = g: [Q′_hi; Q′_lo] for the codes and [Q″_hi; Q″_lo]
        // for the QJL signs, k order following the key decoders' dims.  G4: the same
        // pairs of head hq = g / 2, of which column g of step4's B operand takes the
        // high (g even) or low (g odd) halves.
        const int hq = G4 ? (g >> 1) : g;
        uint32_t AQ[kKB][4], AS[kKB][4];
        {
            const float i1 = 1.f / qsc[hq], i2 = 1.f / qsc[kHeads + hq];
            // this lane's 32 dims of q′ (and q″): chunk c of head hq, eight 16-byte loads
            float q1[32], q2[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 u = *reinterpret_cast<const float4*>(qsh + qidx(hq, 32 * c) + 4 * k);
                q1[4 * k] = u.x;
                q1[4 * k + 1] = u.y;
                q1[4 * k + 2] = u.z;
                q1[4 * k + 3] = u.w;
                if constexpr (KP) {
                    const float4 v = *reinterpret_cast<const float4*>(qsh + kHeads * kQRow + qidx(hq, 32 * c) + 4 * k);
                    q2[4 * k] = v.x;
                    q2[4 * k + 1] = v.y;
                    q2[4 * k + 2] = v.z;
                    q2[4 * k + 3] = v.w;
                }
            }
            // f16 high part of a pair for rows 0–7, its rounding error for rows 8–15
            auto split = [](float x0, float x1, uint32_t& hi, uint32_t& lo) {
                const __half2 hh = __floats2half2_rn(x0, x1);
                const float2 hf = __half22float2(hh);
                hi = *reinterpret_cast<const uint32_t*>(&hh);
                lo = pack_h2(x0 - hf.x, x1 - hf.y);
            };
#pragma unroll
            for (int kb = 0; kb < kKB; ++kb) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // h = 0: k slots 2c, 2c + 1; h = 1: 2c + 8, 2c + 9
                    if constexpr (KB > 0)
                        split(q1[KDecoder<KB>::dim(0, kb, 2 * h)] * i1, q1[KDecoder<KB>::dim(0, kb, 2 * h + 1)] * i1,
                              AQ[kb][2 * h], AQ[kb][2 * h + 1]);
                    else
                        AQ[kb][2 * h] = AQ[kb][2 * h + 1] = 0u;
                    if constexpr (KP)
                        split(q2[ksign_dim(0, kb, 2 * h)] * i2, q2[ksign_dim(0, kb, 2 * h + 1)] * i2, AS[kb][2 * h],
                              AS[kb][2 * h + 1]);
                    else
                        AS[kb][2 * h] = AS[kb][2 * h + 1] = 0u;
                }
            }
        }
        uint32_t BQ[G4 ? kKB : 1][2], BS[G4 ? kKB : 1][2];
        if constexpr (G4) {
            const bool lo = g & 1;
#pragma unroll
            for (int kb = 0; kb < kKB; ++kb) {
                BQ[kb][0] = lo ? AQ[kb][1] : AQ[kb][0];
                BQ[kb][1] = lo ? AQ[kb][3] : AQ[kb][2];
                BS[kb][0] = lo ? AS[kb][1] : AS[kb][0];
                BS[kb][1] = lo ? AS[kb][3] : AS[kb][2];
            }
        }
        // score factors of this lane's head (g; G4: c), log2 units
        const int hs = G4 ? c : g;
        const float scale2 = a.scale * kLog2e;
        const float fK = scale2 * qsc[hs] / a.kcb.lut_scale;
        const float fS = scale2 * a.kgamma * qsc[kHeads + hs];
        KDecoder<KB> dk;
        Decoder<VB> dv;
        dk.init(a.kcb, mp + SM::kTabK, lane);
        dv.init(a.vcb, mp + SM::kTabV, lane);
        SignDecoder ds;
        const uint32_t stab = KP ? KSignTable::lane_base(mp + SM::kTabS, lane) : 0u;

        // ---- consumers: tile t is rows 16·(t mod n) … of stage t / n (n tiles per stage)
        int tile = warp;
        if constexpr (AA) {  // the tiles of the first ns_safe stages (all full) before the wait
            constexpr int kTilesPerStage = ST::R / kTile;
            const int tlim = t0 + ns_safe * ST::R;
            for (; tile < ns_safe * kTilesPerStage; tile += W) {
                const int stage = tile / kTilesPerStage, slot = stage % SM::kStages;
                const bool ok = sm100::mbar_wait(&s_full[slot], (uint32_t)((stage / SM::kStages) & 1), a.status,
                                                 kDecodeStageTimeout);
                if (!__all_sync(0xffffffffu, ok)) {
                    tile = 1 << 30;  // gave up: no further tiles
                    break;
                }
                const int tb = t0 + tile * kTile, r0 = (tile % kTilesPerStage) * kTile;
                const unsigned char* stp = mp + SM::kStage + (size_t)slot * ST::kBytes;
                if constexpr (G4)
                    step4<KB, KP, VB, VP, true>(st, stp, r0, tb, tlim, dk, dv, ds, stab, BQ, BS, fK, fS, a, head0, G, g,
                                                c);
                else
                    step<KB, KP, VB, VP, true>(st, stp, r0, tb, tlim, dk, dv, ds, stab, AQ, AS, fK, fS, a, head0, G, g,
                                               c);
                __syncwarp();
                if (lane == 0) sm100::mbar_arrive(&s_empty[slot]);
            }
            read_length();
        }
        for (; tile < ntiles; tile += W) {
            constexpr int kTilesPerStage = ST::R / kTile;
            const int stage = tile / kTilesPerStage, slot = stage % SM::kStages;
            const bool ok = sm100::mbar_wait(&s_full[slot], (uint32_t)((stage / SM::kStages) & 1), a.status,
                                             kDecodeStageTimeout);
            if (!__all_sync(0xffffffffu, ok)) break;  // the warp gives up together
            const int tb = t0 + tile * kTile, r0 = (tile % kTilesPerStage) * kTile;
            const unsigned char* stp = mp + SM::kStage + (size_t)slot * ST::kBytes;
            if constexpr (G4) {
                if (tb + kTile <= t1)
                    step4<KB, KP, VB, VP, true>(st, stp, r0, tb, t1, dk, dv, ds, stab, BQ, BS, fK, fS, a, head0, G, g, c);
                else
                    step4<KB, KP, VB, VP, false>(st, stp, r0, tb, t1, dk, dv, ds, stab, BQ, BS, fK, fS, a, head0, G, g,
                                                 c);
            } else {
                if (tb + kTile <= t1)
                    step<KB, KP, VB, VP, true>(st, stp, r0, tb, t1, dk, dv, ds, stab, AQ, AS, fK, fS, a, head0, G, g, c);
                else
                    step<KB, KP, VB, VP, false>(st, stp, r0, tb, t1, dk, dv, ds, stab, AQ, AS, fK, fS, a, head0, G, g, c);
            }
            __syncwarp();  // every lane has read the tile before the stage is released
            if (lane == 0) sm100::mbar_arrive(&s_empty[slot]);
        }
    }

    // ---- combine the warps of this CTA into one split partial per head (the lanes
    // holding a head's sum: the quad g, or with G4 the eight lanes of one c)
    if constexpr (G4) {
        st.l += __shfl_xor_sync(0xffffffffu, st.l, 4);
        st.l += __shfl_xor_sync(0xffffffffu, st.l, 8);
        st.l += __shfl_xor_sync(0xffffffffu, st.l, 16);
    } else {
        st.l += __shfl_xor_sync(0xffffffffu, st.l, 1);
        st.l += __shfl_xor_sync(0xffffffffu, st.l, 2);
    }
    __syncthreads();  // tables, queries and rings are dead from here on
    float* wM = reinterpret_cast<float*>(smem + SM::kWM);    // [warp][head] running maxima
    float* wL = reinterpret_cast<float*>(smem + SM::kWL);    // [warp][head] sums
    float* wF = reinterpret_cast<float*>(smem + SM::kWF);    // [warp][head] weights 2^(M_w − max_w M_w)
    float* wO = reinterpret_cast<float*>(smem + SM::kWO);    // [warp][m][i][lane]
    float* wO2 = reinterpret_cast<float*>(smem + SM::kWO2);  // [warp][m][i][lane] (prod values)
    // accumulators in fragment order: each store is 32 consecutive words
    constexpr int kFrag = kMT * 4 * 32;
    if (!producer) {
        if constexpr (G4) {  // heads c from lanes g = 0; heads 4–7 (none) from lanes g = 1
            if (g < 2) {
                wM[warp * kHeads + 4 * g + c] = g == 0 ? st.M : -INFINITY;
                wL[warp * kHeads + 4 * g + c] = g == 0 ? st.l : 0.f;
            }
        } else if (c == 0) {
            wM[warp * kHeads + g] = st.M;
            wL[warp * kHeads + g] = st.l;
        }
#pragma unroll
        for (int m = 0; m < kMT; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                wO[warp * kFrag + (m * 4 + i) * 32 + lane] = st.O[m][i];
                if constexpr (VP) wO2[warp * kFrag + (m * 4 + i) * 32 + lane] = st.O2[m][i];
            }
    }
    __syncthreads();
    if (threadIdx.x < kHeads) {
        const int h = threadIdx.x;
        float Mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) Mx = fmaxf(Mx, wM[w * kHeads + h]);
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const float f = Mx == -INFINITY ? 0.f : ex2(wM[w * kHeads + h] - Mx);
            wF[w * kHeads + h] = f;
            lsum = fmaf(f, wL[w * kHeads + h], lsum);
        }
        if (h < G) {
            const size_t ps = (head0 + h) * a.n_splits + split;
            a.pm[ps] = Mx == -INFINITY ? -INFINITY : Mx * kLn2;
            a.pl[ps] = lsum;
        }
    }
    __syncthreads();
    // element (m, i, lane) of the accumulator fragments: head 2c + (i & 1), dim from the
    // decode map (rows g, g + 8 of m-tile m are element g & 1 of pairs 2m, 2m + 1 of run g >> 1)
    const float inv_vs = 1.f / a.vcb.lut_scale;
    for (int f = threadIdx.x; f < kFrag; f += blockDim.x) {
        const int fl = f & 31, fi = (f >> 5) & 3, fm = f >> 7;
        const int h = 2 * (fl & 3) + (fi & 1), fg = fl >> 2;
        if (h >= G) continue;
        float o = 0.f, o2 = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const float wf = wF[w * kHeads + h];
            o = fmaf(wf, wO[w * kFrag + f], o);
            if constexpr (VP) o2 = fmaf(wf, wO2[w * kFrag + f], o2);
        }
        const size_t ps = (head0 + h) * a.n_splits + split;
        const int tau = 2 * fm + (fi >> 1);
        if constexpr (VB > 0) a.pacc[ps * D + Decoder<VB>::dim(fg >> 1, tau, fg & 1)] = o * inv_vs;
        else a.pacc[ps * D + sign_dim(fg >> 1, tau, fg & 1)] = 0.f;
        if constexpr (VP) a.pacc2[ps * D + sign_dim(fg >> 1, tau, fg & 1)] = o2;
    }

    // ---- the last CTA of this group to finish merges all of its splits: the
    // barrier orders every thread's partial stores before thread 0's ticket, whose
    // acquire-release add publishes them and, in the last CTA, acquires the others'
    __syncthreads();
    if (threadIdx.x == 0) {
        const int group = (b * a.Hkv + kvh) * a.n_hblocks + hb;
        int old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(a.cnt + group) : "memory");
        s_last = old == a.n_splits - 1;
    }
    __syncthreads();
    if (!s_last) return;
    merge_group<KB, KP, VB, VP>(a, smem, head0, G);
}

// pdl: launched as the programmatic dependent of the kernel before it in the
// stream.  That kernel must not write the workspace; with a.after_append it must not
// write q either (the decode-step append), else it may be anything (the ticket
// clearing kernel, which completes only after the kernels before it).
template <int KB, bool KP, int VB, bool VP, bool AA, bool G4>
int launch_split_mma_v(const SplitArgs& a, dim3 grid, bool pdl, cudaStream_t s) {
    using SM = Smem<KB, KP, VB, VP>;
    static_assert(SM::kBytes <= 232448 - 1024, "decode shared memory above the per-CTA limit");
    auto fn = decode_split_mma_kernel<KB, KP, VB, VP, AA, G4>;
    static std::atomic<uint64_t> smem_set{0};
    const int rc = ensure_smem_attr(smem_set, (const void*)fn, (int)SM::kBytes, "decode (tensor-core) smem attribute");
    if (rc != TQ_OK) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(SM::kThreads);
    cfg.dynamicSmemBytes = SM::kBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, a);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "decode (tensor-core) split launch");
}

template <int KB, bool KP, int VB, bool VP>
int launch_split_mma(const SplitArgs& a, dim3 grid, bool pdl, cudaStream_t s) {
    const bool aa = a.after_append && (a.T_max & 3) == 0 && a.chunk >= kAppendStreamChunk, g4 = a.G <= 4;
    if (g4) return aa ? launch_split_mma_v<KB, KP, VB, VP, true, true>(a, grid, pdl, s)
                      : launch_split_mma_v<KB, KP, VB, VP, false, true>(a, grid, pdl, s);
    return aa ? launch_split_mma_v<KB, KP, VB, VP, true, false>(a, grid, pdl, s)
              : launch_split_mma_v<KB, KP, VB, VP, false, false>(a, grid, pdl, s);
}

// Values dispatched at run time for one key configuration (see tq_decode_args.h).
template <int KB, bool KP>
int launch_for_k(const SplitArgs& a, dim3 grid, int vb, bool vp, bool pdl, cudaStream_t s) {
    if (vp) {
        switch (vb) {
            case 0: return launch_split_mma<KB, KP, 0, true>(a, grid, pdl, s);
            case 1: return launch_split_mma<KB, KP, 1, true>(a, grid, pdl, s);
            case 2: return launch_split_mma<KB, KP, 2, true>(a, grid, pdl, s);
            case 3: return launch_split_mma<KB, KP, 3, true>(a, grid, pdl, s);
            default: break;
        }
    } else {
        switch (vb) {
            case 1: return launch_split_mma<KB, KP, 1, false>(a, grid, pdl, s);
            case 2: return launch_split_mma<KB, KP, 2, false>(a, grid, pdl, s);
            case 3: return launch_split_mma<KB, KP, 3, false>(a, grid, pdl, s);
            case 4: return launch_split_mma<KB, KP, 4, false>(a, grid, pdl, s);
            default: break;
        }
    }
    return fail(TQ_EUNSUPPORTED, "tensor-core decode: value b_m=%d", vb);
}

}  // namespace mmadec
}  // namespace tq
