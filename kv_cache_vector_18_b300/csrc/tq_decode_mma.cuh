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
// 16-token step, lane = 4·g + c:
//   scores  S[16 tokens × 8 heads] = K̃[16 × d] · Q′ᵀ[d × 8]: the A fragment is
//           decoded in registers straight from the packed codes — lane (g, c)
//           owns tokens g and g + 8 and the 32 dims [32c, 32c + 32) of each, so
//           its code bits are one contiguous run of the row.  Four (or two)
//           consecutive codes index a shared-memory table of f16 centroid pairs;
//           one byte of QJL sign bits indexes a table of four ±1 pairs.  Table
//           words are read one 32-bit load per fragment register, so each lands
//           directly in its MMA operand slot.  Q′ (and Q″ = S·q) are B fragments
//           whose k order follows the decoded pairs.
//   values  Oᵀ[d × 8 heads] += Ṽᵀ[d × 16 tokens] · P′ᵀ[16 × 8]: Ṽ is decoded the
//           same way (token-major pairs) and moved to the dim-major A layout
//           with movmatrix.trans; P′ leaves the score accumulator in exactly the
//           layout movmatrix.trans turns into the B fragment.
// ‖v_t‖ is folded into the softmax exponent (P′_t = 2^(s_t·log2e + log2‖v_t‖ − M)),
// so the f16 weights stay bounded whatever the value norms; l accumulates
// P′_t/‖v_t‖ in f32 against the same running maximum M.  M is raised only when a
// step's exponent exceeds it by more than kSlack, so P′ ≤ 2^kSlack and most
// steps skip the cross-lane maximum.  Per-head scale factors keep the f16 query
// fragments in [−1, 1], and the centroid tables hold f16(σ·c) for a per-codebook
// σ chosen on the host so that the f16 rounding of the centroids — systematic,
// and amplified by the softmax — nearly vanishes.
//
// Data movement: each warp streams its 16-token tiles of all packed planes into
// a two-stage shared-memory ring with cp.async (the next tile is in flight while
// the current one is decoded), so the hot loop reads its operands with short
// shared-memory loads.  The last CTA of each (batch, KV head, head block) to
// finish merges every split's partial and applies Π_vᵀ (no merge launch).
#pragma once

#include <math.h>

#include "tq_common.cuh"
#include "tq_decode_args.h"

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

// ---- per-lane decoders: packed codes → f16 fragment pairs -------------------
// A lane owns a run of 32 consecutive codes of a row (dims [32c, 32c + 32)).
// Decoder<B>::pairs(w, kb, p0, p1) yields the two f16 pairs that k16 block kb
// of an MMA fragment takes from that run (pairs τ = 2kb and 2kb + 1), and
// Decoder<B>::dim(c, τ, e) is the dim held by element e of pair τ — the Q′
// fragments and the accumulator rows follow the same map.
//   B = 1: both codes of a pair are bits τ and τ + 16 of the run's word; the
//          centroids are ±c₁, so the pair is the constant (−c₁, −c₁) with its
//          two sign bits flipped where the code bits are set (two ALU ops).
//   B = 2: a shared-memory table indexed by four adjacent codes (one byte)
//          whose entry is the two f16 pairs, 16 interleaved copies so that a
//          warp's lookups never collide on a bank.
//   B = 3, 4: a shared-memory table of f16 centroid pairs indexed by two
//          adjacent codes, one copy per lane.
// (Measured on B300 against register-only variants — byte permutes for B = 2,
// two bit operations per QJL sign pair — the tables are faster: the integer
// pipe, not shared memory, is the tighter resource.)
__device__ __forceinline__ uint32_t flip_pair(uint32_t w, int tau, uint32_t neg) {
    return neg ^ ((w << (15 - tau)) & 0x80008000u);
}

template <int B>
struct Decoder {
    static constexpr bool kQuadTable = B == 2;  // 256 quads × 16 copies × 8 bytes
    static constexpr bool kTable = B >= 3;
    static constexpr size_t kTableBytes =
        kTable ? (size_t)(1 << (2 * B)) * 32 * 4 : (kQuadTable ? (size_t)256 * 16 * 8 : 0);
    static constexpr int kWords = B > 0 ? B : 1;
    // per-lane constants
    uint32_t k0, k1;   // B = 1: (−c₁, −c₁); B = 2: levels (c0, c1), (c2, c3); B ≥ 3: table base | lane offset
    uint32_t tab;

    __device__ static void fill(unsigned char* tabp, const Codebook& cb) {
        if constexpr (kQuadTable) {
            const float s = cb.lut_scale;
            for (int i = threadIdx.x; i < 256 * 16; i += blockDim.x) {
                const uint32_t e = (uint32_t)i >> 4, copy = (uint32_t)i & 15u;
                uint2 v;
                v.x = pack_h2(cb.c[e & 3] * s, cb.c[(e >> 2) & 3] * s);
                v.y = pack_h2(cb.c[(e >> 4) & 3] * s, cb.c[(e >> 6) & 3] * s);
                *reinterpret_cast<uint2*>(tabp + e * 128u + copy * 8u) = v;
            }
        }
        if constexpr (kTable) {
            const float s = cb.lut_scale;
            constexpr uint32_t m = (1u << B) - 1u;
            for (int i = threadIdx.x; i < (1 << (2 * B)) * 32; i += blockDim.x) {
                const uint32_t e = (uint32_t)i >> 5, copy = (uint32_t)i & 31u;
                *reinterpret_cast<uint32_t*>(tabp + e * 128u + copy * 4u) =
                    pack_h2(cb.c[e & m] * s, cb.c[(e >> B) & m] * s);
            }
        }
    }
    __device__ void init(const Codebook& cb, const unsigned char* tabp, int lane) {
        const float s = cb.lut_scale;
        if constexpr (B == 1) {
            k0 = pack_h2(cb.c[0] * s, cb.c[0] * s);
        } else if constexpr (kQuadTable) {
            tab = smem_addr(tabp) + (uint32_t)(lane & 15) * 8u;
        } else if constexpr (B == 2) {
            k0 = pack_h2(cb.c[0] * s, cb.c[1] * s);
            k1 = pack_h2(cb.c[2] * s, cb.c[3] * s);
        } else if constexpr (kTable) {
            tab = smem_addr(tabp) + (uint32_t)lane * 4u;
        }
    }
    __device__ __forceinline__ void pairs(const uint32_t* w, int kb, uint32_t& p0, uint32_t& p1) const {
        if constexpr (B == 1) {
            p0 = flip_pair(w[0], 2 * kb, k0);
            p1 = flip_pair(w[0], 2 * kb + 1, k0);
        } else if constexpr (kQuadTable) {
            const uint32_t a = field_off<8, 7>(w, 8 * kb) | tab;
            p0 = lds32(a);
            p1 = lds32o<4>(a);
        } else if constexpr (B == 2) {
            const int wi = kb >> 2, j = kb & 3;
            const uint32_t x = (w[wi] >> (2 * j)) & 0x03030303u;  // codes j, j+4, j+8, j+12 in bytes
            const uint32_t y = x * 0x22u + 0x10101010u;           // byte-permute selectors
            p0 = __byte_perm(k0, k1, y);
            p1 = __byte_perm(k0, k1, y >> 16);
        } else {
            p0 = lds32(field_off<2 * B, 7>(w, 4 * B * kb) | tab);
            p1 = lds32(field_off<2 * B, 7>(w, 4 * B * kb + 2 * B) | tab);
        }
    }
    __host__ __device__ static constexpr int dim(int c, int tau, int e) {
        return B == 1 ? 32 * c + tau + 16 * e
                      : ((B == 2 && !kQuadTable) ? 32 * c + 16 * ((tau >> 1) >> 2) + ((tau >> 1) & 3) + 8 * (tau & 1) +
                                                       4 * e
                                                 : 32 * c + 2 * tau + e);
    }
};

constexpr uint32_t kMinusOnePair = 0xBC00BC00u;  // f16 (−1, −1)

// Every table is placed at a shared-memory address that is a multiple of its
// (power-of-two) size, so a lookup address is one OR of the shifted code field
// with the lane's copy offset and the table base.

// QJL sign pairs of a lane's 32 sign bits: either two ALU operations per pair
// (bits τ, τ + 16), or a shared-memory table mapping one byte of sign bits to
// four ±1 pairs (bits 2τ, 2τ + 1), 8 copies so that lookups never collide.
struct SignDecoder {
    static constexpr bool kTable = true;
    static constexpr size_t kTableBytes = kTable ? (size_t)256 * 8 * 16 : 0;
    uint32_t tab;
    __device__ static void fill(unsigned char* tabp) {
        if constexpr (kTable) {
            for (int i = threadIdx.x; i < 256 * 8; i += blockDim.x) {
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
    }
    __device__ void init(const unsigned char* tabp, int lane) {
        if constexpr (kTable) tab = smem_addr(tabp) + (uint32_t)(lane & 7) * 16u;
    }
    // pairs 4m..4m+3 (k16 blocks 2m and 2m + 1)
    __device__ __forceinline__ void quad(uint32_t w, int m, uint32_t (&p)[4]) const {
        if constexpr (kTable) {
            const uint32_t a = field_off<8, 7>(&w, 8 * m) | tab;
            p[0] = lds32(a);
            p[1] = lds32o<4>(a);
            p[2] = lds32o<8>(a);
            p[3] = lds32o<12>(a);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = flip_pair(w, 4 * m + i, kMinusOnePair);
        }
    }
    __host__ __device__ static constexpr int dim(int c, int tau, int e) {
        return kTable ? 32 * c + 2 * tau + e : 32 * c + tau + 16 * e;
    }
};
__host__ __device__ constexpr int sign_dim(int c, int tau, int e) { return SignDecoder::dim(c, tau, e); }

// Byte layout of one 16-token tile of every plane in a warp's staging ring.
template <int KB, bool KP, int VB, bool VP>
struct Stage {
    static constexpr int kRK = KB * 16, kRV = VB * 16;  // code bytes per row
    static constexpr int kKC = 0;
    static constexpr int kKS = kKC + kTile * kRK;
    static constexpr int kKN = kKS + (KP ? kTile * 16 : 0);
    static constexpr int kKR = kKN + kTile * 4;
    static constexpr int kVC = kKR + (KP ? kTile * 4 : 0);
    static constexpr int kVS = kVC + kTile * kRV;
    static constexpr int kVN = kVS + (VP ? kTile * 16 : 0);
    static constexpr int kVR = kVN + kTile * 4;
    static constexpr int kBytes = kVR + (VP ? kTile * 4 : 0);
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

// Rows [tb, tb + 16) of a plane with RB-byte rows (a multiple of 16) into smem
// at dst, chunk k of 16 bytes through lane k mod 32.  `src` is the tile's first
// byte.  A full tile copies without predicates; in the chunk's last tile the
// rows at or past `rows` (tile-relative) are zero-filled without being read.
template <int RB>
__device__ __forceinline__ void stage_rows16(uint32_t dst, const uint8_t* src, bool full, int rows, int lane) {
#pragma unroll
    for (int r = 0; r < (RB + 31) / 32; ++r) {
        const int k = lane + 32 * r;
        if (RB % 32 == 0 || k < RB) {
            if (full) {
                cp_async16(dst + 16 * k, src + 16 * k, 16u);
            } else {
                const bool ok = (16 * k) / RB < rows;
                cp_async16(dst + 16 * k, ok ? src + 16 * k : src, ok ? 16u : 0u);
            }
        }
    }
}
// A tile of fp32 norms: four 16-byte copies (lanes 0–3) when the tile is full and
// the plane's rows start on a 16-byte boundary (a16, uniform over the CTA), else
// one 4-byte copy per row (lanes 0–15).
__device__ __forceinline__ void stage_rows4(uint32_t dst, const float* src, bool full, bool a16, int rows, int lane) {
    if (full && a16) {
        if (lane < 4) cp_async16(dst + 16 * lane, src + 4 * lane, 16u);
    } else if (lane < kTile) {
        const bool ok = full || lane < rows;
        cp_async4(dst + 4 * lane, ok ? src + lane : src, ok ? 4u : 0u);
    }
}

template <int KB, bool KP, int VB, bool VP>
__device__ __forceinline__ void stage_tile(uint32_t dst, const Slab& s, int tb, int t1, int lane) {
    using ST = Stage<KB, KP, VB, VP>;
    const bool full = tb + kTile <= t1;
    const int rows = t1 - tb;
    if constexpr (KB > 0) stage_rows16<ST::kRK>(dst + ST::kKC, s.kc + (size_t)tb * ST::kRK, full, rows, lane);
    if constexpr (KP) {
        stage_rows16<16>(dst + ST::kKS, s.ks + (size_t)tb * 16, full, rows, lane);
        stage_rows4(dst + ST::kKR, s.krn + tb, full, s.a16, rows, lane);
    }
    stage_rows4(dst + ST::kKN, s.kn + tb, full, s.a16, rows, lane);
    if constexpr (VB > 0) stage_rows16<ST::kRV>(dst + ST::kVC, s.vc + (size_t)tb * ST::kRV, full, rows, lane);
    if constexpr (VP) {
        stage_rows16<16>(dst + ST::kVS, s.vs + (size_t)tb * 16, full, rows, lane);
        stage_rows4(dst + ST::kVR, s.vrn + tb, full, s.a16, rows, lane);
    }
    stage_rows4(dst + ST::kVN, s.vn + tb, full, s.a16, rows, lane);
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


// Warps per CTA: 16 (two KV tiles of data in flight per warp, one CTA per SM);
// prod values carry a second accumulator set and run 8 warps with more registers.
template <bool VP>
struct Warps {
    static constexpr int value = VP ? 8 : 16;
};

// The Q″ fragments stay in shared memory (one uint2 per lane and k16 block)
// when registers are short.
template <bool KP, bool VP>
struct QsInSmem {
    static constexpr bool value = KP && !VP;
};

template <int KB, bool KP, int VB, bool VP>
struct Smem {
    static constexpr int W = Warps<VP>::value;
    // main phase: decode tables, queries, query scales, Q″ fragments, staging rings
    // tables (power-of-two sizes) largest first from a 32 KB-aligned base, so that
    // each one starts at a multiple of its own size
    static constexpr size_t kSzK = Decoder<KB>::kTableBytes, kSzV = Decoder<VB>::kTableBytes;
    static constexpr size_t kSzS = (KP || VP) ? SignDecoder::kTableBytes : 0;
    static constexpr size_t kBig = 32768;
    static constexpr size_t table_offset(int which) {  // 0 = keys, 1 = values, 2 = signs
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
    static constexpr size_t kQSf = kQsc + 2 * kHeads * 4;
    static constexpr size_t kQKl = kQSf + (KP ? (size_t)kKB * 32 * 8 : 0);  // [kKB][32] f16 low parts of Q′
    static constexpr size_t kQin = kQKl + (KB > 0 ? (size_t)kKB * 32 * 8 : 0);  // [kHeads][D] raw queries
    static constexpr size_t kStage = (kQin + (size_t)kHeads * D * 4 + 127) & ~(size_t)127;
    static constexpr size_t kMain = kStage + (size_t)W * 2 * Stage<KB, KP, VB, VP>::kBytes;
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
    static constexpr size_t kMO = kML + kHeads * 4;                       // [2][D][kHeads] merged acc
    static constexpr size_t kMP = (kMO + 2 * (size_t)kHeads * D * 4 + 15) & ~(size_t)15;  // [D][D] Π_v, then S_v
    static constexpr size_t kMQ = kMP + (VP ? 2 : 1) * (size_t)D * D * 4;  // [4][kHeads][D] mat-vec partials
    static constexpr size_t kMerge = kMQ + 4 * (size_t)kHeads * D * 4;
    static constexpr size_t kAlignSlack = kBig - 16;  // the 32 KB-aligned base lies at most this far in
    static constexpr size_t kBytes0 = kMain + kAlignSlack > kCombine ? kMain + kAlignSlack : kCombine;
    static constexpr size_t kBytes = kBytes0 > kMerge ? kBytes0 : kMerge;
};

// Per-warp running state of the online softmax (heads 2c, 2c+1 of the lane)
// and the value accumulators.
template <bool VP>
struct Acc {
    float O[kMT][4];
    float O2[VP ? kMT : 1][4];
    float M[2], Mt[2], l[2];
};

template <int KB, bool KP, int VB, bool VP>
__device__ __forceinline__ void step(Acc<VP>& st, const unsigned char* stp, int tb, int t1,
                                     const Decoder<KB>& dk, const Decoder<VB>& dv, const SignDecoder& ds,
                                     const uint32_t (&QK)[kKB][2],
                                     const uint32_t (&QS)[kKB][2], const uint2* qsf, const uint2* qkl, int lane,
                                     const float (&fK)[2],
                                     const float (&fS)[2], const SplitArgs& a, size_t head0, int G, int g, int c) {
    using ST = Stage<KB, KP, VB, VP>;
    const bool vA = tb + g < t1, vB = tb + 8 + g < t1;
    // staged words are read where they are used, to keep few registers live
    auto kwords = [&](int i, uint32_t* w) { read_words<KB>(w, stp + ST::kKC + (g + 8 * i) * ST::kRK + c * (KB * 4)); };
    auto vwords = [&](int i, uint32_t* w) { read_words<VB>(w, stp + ST::kVC + (g + 8 * i) * ST::kRV + c * (VB * 4)); };
    auto word = [&](int off, int i) { return *reinterpret_cast<const uint32_t*>(stp + off + (g + 8 * i) * 16 + c * 4); };
    auto norm = [&](int off, int i) { return *reinterpret_cast<const float*>(stp + off + (g + 8 * i) * 4); };

    // ---- scores: S1 = K̃·Q′ᵀ (codes), S2 = Z·Q″ᵀ (QJL signs)
    float S1[4] = {0.f, 0.f, 0.f, 0.f}, S2[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (KB > 0) {
        uint32_t kwA[KB], kwB[KB];
        kwords(0, kwA);
        kwords(1, kwB);
#pragma unroll
        for (int kb = 0; kb < kKB; ++kb) {
            uint32_t a0, a1, a2, a3;
            dk.pairs(kwA, kb, a0, a2);
            dk.pairs(kwB, kb, a1, a3);
            mma16816(S1, a0, a1, a2, a3, QK[kb][0], QK[kb][1]);
            const uint2 lo = qkl[kb * 32 + lane];  // Q′ − f16(Q′): the score keeps ~2⁻²² of q′
            mma16816(S1, a0, a1, a2, a3, lo.x, lo.y);
        }
    }
    if constexpr (KP) {
        const uint32_t ksA = word(ST::kKS, 0), ksB = word(ST::kKS, 1);
#pragma unroll
        for (int m = 0; m < kKB / 2; ++m) {
            uint32_t pa[4], pb[4];
            ds.quad(ksA, m, pa);
            ds.quad(ksB, m, pb);
            uint2 q0, q1;
            if constexpr (QsInSmem<KP, VP>::value) {
                q0 = qsf[(2 * m) * 32 + lane];
                q1 = qsf[(2 * m + 1) * 32 + lane];
            } else {
                q0 = make_uint2(QS[2 * m][0], QS[2 * m][1]);
                q1 = make_uint2(QS[2 * m + 1][0], QS[2 * m + 1][1]);
            }
            mma16816(S2, pa[0], pb[0], pa[1], pb[1], q0.x, q0.y);
            mma16816(S2, pa[2], pb[2], pa[3], pb[3], q1.x, q1.y);
        }
    }
    // C layout: [0] (token g, head 2c) [1] (g, 2c+1) [2] (g+8, 2c) [3] (g+8, 2c+1)
    // z = s·log2e + log2‖v‖ (the exponent of the value weight), −∞ past the chunk
    const float vnA = fmaxf(norm(ST::kVN, 0), 1e-30f), vnB = fmaxf(norm(ST::kVN, 1), 1e-30f);
    const float knr[2] = {norm(ST::kKN, 0), norm(ST::kKN, 1)};
    float krr[2] = {0.f, 0.f};
    if constexpr (KP) {
        krr[0] = norm(ST::kKR, 0);
        krr[1] = norm(ST::kKR, 1);
    }
    const float lvA = lg2(vnA), lvB = lg2(vnB);
    const float rvA = rcp(vnA), rvB = rcp(vnB);
    float z[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int tk = i >> 1, e = i & 1;
        float v = fK[e] * S1[i];
        if constexpr (KP) v = fmaf(fS[e] * krr[tk], S2[i], v);
        z[i] = fmaf(knr[tk], v, tk ? lvB : lvA);
    }
    if (!vA) z[0] = z[1] = -INFINITY;
    if (!vB) z[2] = z[3] = -INFINITY;
    if (a.scores != nullptr) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = tb + g + 8 * (i >> 1), h = 2 * c + (i & 1);
            if (((i >> 1) ? vB : vA) && h < G)
                a.scores[(head0 + h) * a.T_max + t] = (z[i] - ((i >> 1) ? lvB : lvA)) * kLn2;
        }
    }

    // ---- online softmax with a lazily raised maximum
    const bool raise = fmaxf(z[0], z[2]) > st.Mt[0] || fmaxf(z[1], z[3]) > st.Mt[1];
    if (__any_sync(0xffffffffu, raise)) {
        float corr[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float mx = fmaxf(z[e], z[2 + e]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float Mn = fmaxf(st.M[e], mx);
            corr[e] = ex2(st.M[e] - Mn);  // 0 on the first step (M = −∞)
            st.M[e] = Mn;
            st.Mt[e] = Mn + kSlack;
            st.l[e] *= corr[e];
        }
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
            st.O[m][0] *= corr[0];
            st.O[m][1] *= corr[1];
            st.O[m][2] *= corr[0];
            st.O[m][3] *= corr[1];
            if constexpr (VP) {
                st.O2[m][0] *= corr[0];
                st.O2[m][1] *= corr[1];
                st.O2[m][2] *= corr[0];
                st.O2[m][3] *= corr[1];
            }
        }
    }
    float pv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = i & 1;
        pv[i] = ex2(z[i] - st.M[e]);
        st.l[e] = fmaf(pv[i], (i >> 1) ? rvB : rvA, st.l[e]);
    }
    const uint32_t PB0 = mov_trans(pack_h2(pv[0], pv[1]));
    const uint32_t PB1 = mov_trans(pack_h2(pv[2], pv[3]));

    // ---- values: Oᵀ += Ṽᵀ·P′ᵀ in the rotated frame
    if constexpr (VB > 0) {
        uint32_t vwA[VB], vwB[VB];
        vwords(0, vwA);
        vwords(1, vwB);
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
            uint32_t x0, x1, y0, y1;
            dv.pairs(vwA, m, x0, x1);
            dv.pairs(vwB, m, y0, y1);
            mma16816(st.O[m], mov_trans(x0), mov_trans(x1), mov_trans(y0), mov_trans(y1), PB0, PB1);
        }
    }
    if constexpr (VP) {
        const float gA = a.vgamma * norm(ST::kVR, 0), gB = a.vgamma * norm(ST::kVR, 1);
        const uint32_t vsA = word(ST::kVS, 0), vsB = word(ST::kVS, 1);
        const uint32_t QB0 = mov_trans(pack_h2(pv[0] * gA, pv[1] * gA));
        const uint32_t QB1 = mov_trans(pack_h2(pv[2] * gB, pv[3] * gB));
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
    constexpr int NT = SM::W * 32;
    float* wts = reinterpret_cast<float*>(smem + SM::kMW);   // [kHeads][kMaxSplits]
    float* linv = reinterpret_cast<float*>(smem + SM::kML);  // [kHeads]
    float* mo = reinterpret_cast<float*>(smem + SM::kMO);    // [2][D][kHeads]
    float* pis = reinterpret_cast<float*>(smem + SM::kMP);   // [D][D] Π_v, then [D][D] S_v
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ns = a.n_splits;
    // stage Π_v (and S_v) while the split weights are formed: all loads in flight at once
#pragma unroll
    for (int i = threadIdx.x; i < D * D / 4; i += NT)
        reinterpret_cast<float4*>(pis)[i] = __ldg(reinterpret_cast<const float4*>(a.vPi) + i);
    if constexpr (VP) {
#pragma unroll
        for (int i = threadIdx.x; i < D * D / 4; i += NT)
            reinterpret_cast<float4*>(pis + D * D)[i] = __ldg(reinterpret_cast<const float4*>(a.vS) + i);
    }
    if (warp < G) {
        const size_t hs = (head0 + warp) * ns;
        float mx = -INFINITY;
        for (int s = lane; s < ns; s += 32) mx = fmaxf(mx, __ldcg(a.pm + hs + s));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float l = 0.f;
        for (int s = lane; s < ns; s += 32) {
            const float f = mx == -INFINITY ? 0.f : ex2((__ldcg(a.pm + hs + s) - mx) * kLog2e);
            wts[warp * SM::kMaxSplits + s] = f;
            l = fmaf(f, __ldcg(a.pl + hs + s), l);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) linv[warp] = l > 0.f ? 1.f / l : 0.f;
    }
    __syncthreads();
    // Σ over splits, coalesced over dims (up to 32 splits' loads in flight per
    // round); stored dim-major so the mat-vec reads the 8 heads of a dim at once
    for (int i = threadIdx.x; i < G * D; i += NT) {
        const int h = i / D, j = i % D;
        const size_t hs = (head0 + h) * ns;
        const float* w = wts + h * SM::kMaxSplits;
        float o = 0.f, o2 = 0.f;
        for (int s0 = 0; s0 < ns; s0 += 32) {
            float v[32], v2[VP ? 32 : 1];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const bool in = s0 + k < ns;
                v[k] = in ? __ldcg(a.pacc + (hs + s0 + k) * D + j) : 0.f;
                if constexpr (VP) v2[k] = in ? __ldcg(a.pacc2 + (hs + s0 + k) * D + j) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float wk = s0 + k < ns ? w[s0 + k] : 0.f;
                o = fmaf(wk, v[k], o);
                if constexpr (VP) o2 = fmaf(wk, v2[k], o2);
            }
        }
        mo[j * kHeads + h] = o * linv[h];
        if constexpr (VP) mo[kHeads * D + j * kHeads + h] = o2 * linv[h];
    }
    for (int i = G * D + threadIdx.x; i < kHeads * D; i += NT) {  // heads past G: zero
        mo[(i % D) * kHeads + i / D] = 0.f;
        if constexpr (VP) mo[kHeads * D + (i % D) * kHeads + i / D] = 0.f;
    }
    __syncthreads();
    // out[h][col] = Σ_j Π_v[j][col]·o[j][h] (+ S_v[j][col]·o2[j][h]): thread (col, quarter)
    // sums its quarter of j for all 8 heads (one matrix load feeds 8 FMAs), then
    // the four quarters are added
    float* part = reinterpret_cast<float*>(smem + SM::kMQ);  // [4][kHeads][D]
    for (int t2 = threadIdx.x; t2 < 4 * D; t2 += NT) {
        const int col = t2 % D, jq = t2 / D;
        float r[kHeads];
#pragma unroll
        for (int k = 0; k < kHeads; ++k) r[k] = 0.f;
#pragma unroll
        for (int mtx = 0; mtx < (VP ? 2 : 1); ++mtx) {
            const float* P = pis + mtx * D * D;
            const float* Mo = mo + mtx * kHeads * D;
#pragma unroll 4
            for (int j = 32 * jq; j < 32 * jq + 32; ++j) {
                const float p = P[j * D + col];
                const float4 m0 = *reinterpret_cast<const float4*>(Mo + j * kHeads);
                const float4 m1 = *reinterpret_cast<const float4*>(Mo + j * kHeads + 4);
                r[0] = fmaf(p, m0.x, r[0]);
                r[1] = fmaf(p, m0.y, r[1]);
                r[2] = fmaf(p, m0.z, r[2]);
                r[3] = fmaf(p, m0.w, r[3]);
                r[4] = fmaf(p, m1.x, r[4]);
                r[5] = fmaf(p, m1.y, r[5]);
                r[6] = fmaf(p, m1.z, r[6]);
                r[7] = fmaf(p, m1.w, r[7]);
            }
        }
#pragma unroll
        for (int k = 0; k < kHeads; ++k) part[(jq * kHeads + k) * D + col] = r[k];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * D; i += NT) {
        const int h = i / D, col = i % D;
        a.out[(head0 + h) * D + col] = (part[(0 * kHeads + h) * D + col] + part[(1 * kHeads + h) * D + col]) +
                                       (part[(2 * kHeads + h) * D + col] + part[(3 * kHeads + h) * D + col]);
    }
}

template <int KB, bool KP, int VB, bool VP>
__global__ void __launch_bounds__(Warps<VP>::value * 32, 1) decode_split_mma_kernel(const SplitArgs a) {
    using SM = Smem<KB, KP, VB, VP>;
    using ST = Stage<KB, KP, VB, VP>;
    constexpr int W = SM::W;
    extern __shared__ __align__(128) unsigned char smem[];
    // main-phase regions start at the first 32 KB-aligned shared address
    const uint32_t sbase = smem_addr(smem);
    unsigned char* mp = smem + (((sbase + (uint32_t)SM::kBig - 1u) & ~((uint32_t)SM::kBig - 1u)) - sbase);
    float* qsh = reinterpret_cast<float*>(mp + SM::kQ);     // [2][kHeads][kQRow]: q′, q″ (see qidx)
    float* qsc = reinterpret_cast<float*>(mp + SM::kQsc);   // [2][kHeads]
    uint2* qsf = reinterpret_cast<uint2*>(mp + SM::kQSf);    // [kKB][32]
    uint2* qkl = reinterpret_cast<uint2*>(mp + SM::kQKl);    // [kKB][32]
    __shared__ int s_last;

    const int hb = blockIdx.y % a.n_hblocks, kvh = blockIdx.y / a.n_hblocks;
    const int G = min(kHeads, a.G - hb * kHeads);
    const int split = blockIdx.x, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    int L = a.seq_lens[b];
    L = L < 0 ? 0 : (L > a.T_max ? a.T_max : L);
    const int t0 = split * a.chunk;
    const int t1 = min(t0 + a.chunk, L);
    const size_t head0 = (size_t)b * a.Hq + (size_t)kvh * a.G + (size_t)hb * kHeads;
    const int64_t rowbase = ((int64_t)b * a.Hkv + kvh) * a.T_max;

    // Π_v (and S_v) of the final merge: one L2 prefetch per 128-byte line, spread
    // over the CTAs of the grid, kept with the evict-last priority
    {
        const int nct = gridDim.x * gridDim.y * gridDim.z;
        const int cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        constexpr int kLines = D * D * 4 / 128;
        const int l = cta + nct * (int)threadIdx.x;
        if (l < (VP ? 2 : 1) * kLines) {
            const float* p = l < kLines ? a.vPi + 32 * l : a.vS + 32 * (l - kLines);
            asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p));
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

    // start streaming this warp's first tile before the prologue
    const int ntiles = t1 > t0 ? (t1 - t0 + kTile - 1) / kTile : 0;
    const uint32_t ring = smem_addr(mp + SM::kStage) + (uint32_t)(warp * 2 * ST::kBytes);
    if (warp < ntiles) stage_tile<KB, KP, VB, VP>(ring, sl, t0 + warp * kTile, t1, lane);
    cp_async_commit();

    // ---- prologue: decode tables, queries, query scales
    // raw queries of this head block: loads issued before the table fill, stored after
    constexpr int NT = W * 32, kQPer = kHeads * D / NT;
    float qv[kQPer];
#pragma unroll
    for (int r = 0; r < kQPer; ++r) {
        const int i = threadIdx.x + r * NT, h = i / D;
        const size_t gi = (head0 + h) * D + (i % D);
        qv[r] = h < G ? (a.q_f32 ? __ldg(static_cast<const float*>(a.q) + gi)
                                 : __bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[gi]))
                      : 0.f;
    }
    Decoder<KB>::fill(mp + SM::kTabK, a.kcb);
    Decoder<VB>::fill(mp + SM::kTabV, a.vcb);
    if constexpr (KP || VP) SignDecoder::fill(mp + SM::kTabS);
    float* qin = reinterpret_cast<float*>(mp + SM::kQin);  // [kHeads][D]
#pragma unroll
    for (int r = 0; r < kQPer; ++r) qin[threadIdx.x + r * NT] = qv[r];
    __syncthreads();
    // q′ = Π_k·q and q″ = S_k·q on the tensor cores: D[16 × 8 dims] = A·B with
    // A = [bf16 hi of the 8 heads' q; bf16 lo] and B = a bf16 half of the matrix,
    // so q_hi·M + q_lo·M is the sum of rows g and g + 8; hi and lo halves of M
    // accumulate in the same tile (fp32-level accuracy).  The contraction order
    // is permuted so that in k16 blocks 2p and 2p + 1 lane (g, c) holds the eight
    // consecutive input dims 32p + 8c … 32p + 8c + 7: its matrix operand is one
    // 16-byte load of row j0 + g.  Each warp takes its 8-dim tiles with all of
    // their loads in flight at once.
    {
        uint32_t A[kKB][4];
#pragma unroll
        for (int ks = 0; ks < kKB; ++ks) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int d0 = 32 * (ks >> 1) + 8 * c + 4 * (ks & 1) + 2 * hh;
                const float2 x = *reinterpret_cast<const float2*>(qin + g * D + d0);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(x.x, x.y);
                const float2 hf = __bfloat1622float2(hi);
                A[ks][2 * hh] = *reinterpret_cast<const uint32_t*>(&hi);
                A[ks][2 * hh + 1] = pack_bf2(x.x - hf.x, x.y - hf.y);
            }
        }
        constexpr int kJobs = (KP ? 2 : 1) * (D / 8);
        constexpr int kPer = (kJobs + W - 1) / W;  // tiles per warp
        uint4 bh[kPer][kKB / 2], bl[kPer][kKB / 2];  // bf16 dims 32p + 8c … + 7 of row j0 + g
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int job = warp + u * W;
            if (job < kJobs) {
                const int second = job >= D / 8, j0 = 8 * (job % (D / 8));
                const uint4* Mh = reinterpret_cast<const uint4*>(second ? a.kS_hi : a.kPi_hi);
                const uint4* Ml = reinterpret_cast<const uint4*>(second ? a.kS_lo : a.kPi_lo);
                const int row = ((j0 + g) * D + 8 * c) >> 3;  // 16-byte index of (j0 + g, 8c)
#pragma unroll
                for (int p2 = 0; p2 < kKB / 2; ++p2) {
                    bh[u][p2] = __ldg(Mh + row + 4 * p2);
                    bl[u][p2] = __ldg(Ml + row + 4 * p2);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int job = warp + u * W;
            if (job < kJobs) {
                const int second = job >= D / 8, j0 = 8 * (job % (D / 8));
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < kKB; ++ks) {
                    const uint4 h = bh[u][ks >> 1], l = bl[u][ks >> 1];
                    mma16816_bf16(acc, A[ks], (ks & 1) ? h.z : h.x, (ks & 1) ? h.w : h.y);
                    mma16816_bf16(acc, A[ks], (ks & 1) ? l.z : l.x, (ks & 1) ? l.w : l.y);
                }
                float* o = qsh + (second ? kHeads * kQRow : 0) + qidx(g, j0 + 2 * c);
                o[0] = acc[0] + acc[2];
                o[1] = acc[1] + acc[3];
            }
        }
    }
    __syncthreads();
    if (warp < kHeads) {
        // warp w finds max|q′| (and max|q″|) of head w
        float m1 = 0.f, m2 = 0.f;
        for (int j = lane; j < D; j += 32) {
            m1 = fmaxf(m1, fabsf(qsh[qidx(warp, j)]));
            if constexpr (KP) m2 = fmaxf(m2, fabsf(qsh[kHeads * kQRow + qidx(warp, j)]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
            m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
        }
        if (lane == 0) {
            qsc[warp] = m1 > 0.f ? m1 : 1.f;
            qsc[kHeads + warp] = m2 > 0.f ? m2 : 1.f;
        }
    }
    __syncthreads();

    // B fragments of Q′ (and Q″) for head g, k order following the decoded pairs.
    uint32_t QK[kKB][2], QS[kKB][2];
    {
        const float i1 = 1.f / qsc[g], i2 = 1.f / qsc[kHeads + g];
        // this lane's 32 dims of q′ (and q″): chunk c of head g, eight 16-byte loads
        float q1[32], q2[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 u = *reinterpret_cast<const float4*>(qsh + qidx(g, 32 * c) + 4 * k);
            q1[4 * k] = u.x;
            q1[4 * k + 1] = u.y;
            q1[4 * k + 2] = u.z;
            q1[4 * k + 3] = u.w;
            if constexpr (KP) {
                const float4 v = *reinterpret_cast<const float4*>(qsh + kHeads * kQRow + qidx(g, 32 * c) + 4 * k);
                q2[4 * k] = v.x;
                q2[4 * k + 1] = v.y;
                q2[4 * k + 2] = v.z;
                q2[4 * k + 3] = v.w;
            }
        }
#pragma unroll
        for (int kb = 0; kb < kKB; ++kb) {
#pragma unroll
            uint32_t lo[2] = {0u, 0u};
            for (int h = 0; h < 2; ++h) {
                const int tau = 2 * kb + h;
                if constexpr (KB > 0) {
                    // f16 high part for the fragment, f16 low part (the rounding error) for a second MMA
                    const float x0 = q1[Decoder<KB>::dim(0, tau, 0)] * i1, x1 = q1[Decoder<KB>::dim(0, tau, 1)] * i1;
                    const __half2 hh = __floats2half2_rn(x0, x1);
                    const float2 hf = __half22float2(hh);
                    QK[kb][h] = *reinterpret_cast<const uint32_t*>(&hh);
                    lo[h] = pack_h2(x0 - hf.x, x1 - hf.y);
                } else {
                    QK[kb][h] = 0u;
                }
                QS[kb][h] = KP ? pack_h2(q2[sign_dim(0, tau, 0)] * i2, q2[sign_dim(0, tau, 1)] * i2) : 0u;
            }
            if constexpr (QsInSmem<KP, VP>::value)
                if (warp == 0) qsf[kb * 32 + lane] = make_uint2(QS[kb][0], QS[kb][1]);
            if constexpr (KB > 0)
                if (warp == 0) qkl[kb * 32 + lane] = make_uint2(lo[0], lo[1]);
        }
    }
    __syncthreads();
    // score factors for this lane's two heads (2c, 2c+1), log2 units
    const float scale2 = a.scale * kLog2e;
    float fK[2], fS[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        fK[e] = scale2 * qsc[2 * c + e] / a.kcb.lut_scale;
        fS[e] = scale2 * a.kgamma * qsc[kHeads + 2 * c + e];
    }
    Decoder<KB> dk;
    Decoder<VB> dv;
    dk.init(a.kcb, mp + SM::kTabK, lane);
    dv.init(a.vcb, mp + SM::kTabV, lane);
    SignDecoder ds;
    ds.init(mp + SM::kTabS, lane);

    Acc<VP> st;
#pragma unroll
    for (int m = 0; m < kMT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            st.O[m][i] = 0.f;
            if constexpr (VP) st.O2[m][i] = 0.f;
        }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        st.M[e] = -INFINITY;
        st.Mt[e] = -INFINITY;
        st.l[e] = 0.f;
    }

    // ---- main loop over this warp's tiles: tile k is staged in ring slot k & 1
    int slot = 0;
    for (int tile = warp; tile < ntiles; tile += W) {
        const int tb = t0 + tile * kTile;
        if (tile + W < ntiles) stage_tile<KB, KP, VB, VP>(ring + (slot ^ 1) * ST::kBytes, sl, tb + W * kTile, t1, lane);
        cp_async_commit();
        cp_async_wait<1>();
        __syncwarp();
        step<KB, KP, VB, VP>(st, mp + SM::kStage + (size_t)(warp * 2 + slot) * ST::kBytes, tb, t1, dk, dv, ds, QK,
                             QS, qsf, qkl, lane, fK, fS, a, head0, G, g, c);
        __syncwarp();  // the slot may be refilled once every lane has read it
        slot ^= 1;
    }
    cp_async_wait<0>();

    // ---- combine the warps of this CTA into one split partial per head
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) st.l[e] += __shfl_xor_sync(0xffffffffu, st.l[e], o);
    __syncthreads();  // tables, queries and rings are dead from here on
    float* wM = reinterpret_cast<float*>(smem + SM::kWM);    // [warp][head] running maxima
    float* wL = reinterpret_cast<float*>(smem + SM::kWL);    // [warp][head] sums
    float* wF = reinterpret_cast<float*>(smem + SM::kWF);    // [warp][head] weights 2^(M_w − max_w M_w)
    float* wO = reinterpret_cast<float*>(smem + SM::kWO);    // [warp][m][i][lane]
    float* wO2 = reinterpret_cast<float*>(smem + SM::kWO2);  // [warp][m][i][lane] (prod values)
    if (g == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            wM[warp * kHeads + 2 * c + e] = st.M[e];
            wL[warp * kHeads + 2 * c + e] = st.l[e];
        }
    }
    // accumulators in fragment order: each store is 32 consecutive words
    constexpr int kFrag = kMT * 4 * 32;
#pragma unroll
    for (int m = 0; m < kMT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            wO[warp * kFrag + (m * 4 + i) * 32 + lane] = st.O[m][i];
            if constexpr (VP) wO2[warp * kFrag + (m * 4 + i) * 32 + lane] = st.O2[m][i];
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

    // ---- the last CTA of this group to finish merges all of its splits
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int group = (b * a.Hkv + kvh) * a.n_hblocks + hb;
        s_last = atomicAdd(a.cnt + group, 1) == a.n_splits - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    merge_group<KB, KP, VB, VP>(a, smem, head0, G);
}

template <int KB, bool KP, int VB, bool VP>
int launch_split_mma(const SplitArgs& a, dim3 grid, cudaStream_t s) {
    using SM = Smem<KB, KP, VB, VP>;
    auto fn = decode_split_mma_kernel<KB, KP, VB, VP>;
    static std::atomic<uint64_t> smem_set{0};
    const int rc = ensure_smem_attr(smem_set, (const void*)fn, (int)SM::kBytes, "decode (tensor-core) smem attribute");
    if (rc != TQ_OK) return rc;
    fn<<<grid, SM::W * 32, SM::kBytes, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "decode (tensor-core) split launch");
}

// Values dispatched at run time for one key configuration (see tq_decode_args.h).
template <int KB, bool KP>
int launch_for_k(const SplitArgs& a, dim3 grid, int vb, bool vp, cudaStream_t s) {
    if (vp) {
        switch (vb) {
            case 0: return launch_split_mma<KB, KP, 0, true>(a, grid, s);
            case 1: return launch_split_mma<KB, KP, 1, true>(a, grid, s);
            case 2: return launch_split_mma<KB, KP, 2, true>(a, grid, s);
            case 3: return launch_split_mma<KB, KP, 3, true>(a, grid, s);
            default: break;
        }
    } else {
        switch (vb) {
            case 1: return launch_split_mma<KB, KP, 1, false>(a, grid, s);
            case 2: return launch_split_mma<KB, KP, 2, false>(a, grid, s);
            case 3: return launch_split_mma<KB, KP, 3, false>(a, grid, s);
            case 4: return launch_split_mma<KB, KP, 4, false>(a, grid, s);
            default: break;
        }
    }
    return fail(TQ_EUNSUPPORTED, "tensor-core decode: value b_m=%d", vb);
}

}  // namespace mmadec
}  // namespace tq
