// Split-K decode attention over a mixed-precision cache on the tensor cores:
// keys and values each split into an outlier part (the 32 channels perm[0..32))
// and the rest (perm[32..128)), each part quantized by its own mse quantizer
// (the page's KV-cache experiment: 32 outlier channels at 3 bits, 96 at 2).
//
// The kernel works in one 128-dim frame per row, [y_o (32 dims); y_n (96 dims)],
// the two parts' rotated coordinates side by side.  With M = blockdiag(Π_o, Π_n)·P
// (P the channel permutation), q′ = M·q and the score of token t is
//   s_t = scale·(‖k_o,t‖·⟨q′_o, c_o[code_o,t]⟩ + ‖k_n,t‖·⟨q′_n, c_n[code_n,t]⟩),
// the value sum Σ_t p_t·[‖v_o,t‖·c_o[code]; ‖v_n,t‖·c_n[code]] in the value
// frame, and the merged output Mᵀ applied to it, scattered back to the
// channels — the same attention the oracle computes on the dequantized rows.
//
// Mapping onto mma.sync.m16n8k16 as in the single-part kernel (tq_decode_mma.cuh),
// with every lane doing the same work: lane (g, c) takes codes 8c … 8c + 7 of
// the outlier part and 24c … 24c + 23 of the rest of its token's row.  k16
// blocks 0–1 of the score hold the outlier part (dims 8c + 4kb + e) and blocks
// 2–7 the rest (dims 32 + 24c + 4(kb − 2) + e), accumulated separately and
// scaled by their own norms; m16 tiles 0–1 of the value product hold the
// outlier part and tiles 2–7 the rest, each weighted by its own value norm.
// The softmax exponent carries log2 of the larger of a token's two value norms,
// so both parts' f16 weights stay below 2^kSlack.
//
// Prod key parts (KP) add each part's QJL term to its score,
// √(π/2)/d_p·‖k_p‖·‖r_p‖·⟨q″_p, z_p⟩ with q″ = blockdiag(S_o, S_n)·P·q: the signs are
// the B operand of a second set of MMAs over the same k16 blocks (lane c takes
// signs 8c … 8c + 7 of the outlier part, one byte, and 24c … 24c + 23 of the rest,
// three bytes, the same dims as its codes), with [Q″_hi; Q″_lo] as A.
#include "tq_decode_mma.cuh"
#include "tq_mixed_decode.h"

namespace tq {
namespace mmadec {
namespace {

constexpr int kDO = 32;        // outlier dims of the frame
constexpr int kDN = D - kDO;   // the rest
constexpr int kMW = 11;        // consumer warps (plus one producer warp)

// Bits [c·NB·8·LEN/8 …) of a row: lane c's run of LEN codes of NB bits, returned
// as NW words (LSB first).  The row starts on a 4-byte boundary; the read may run
// one word past the run (into the next row or plane of the stage).
template <int NB, int LEN, int NW>
__device__ __forceinline__ void lane_run(const unsigned char* row, int c, uint32_t (&r)[NW]) {
    const int bit0 = c * NB * LEN;
    const uint32_t* w = reinterpret_cast<const uint32_t*>(row) + (bit0 >> 5);
    const int sh = bit0 & 31;
    uint32_t cur = w[0];
#pragma unroll
    for (int k = 0; k < NW; ++k) {
        const uint32_t nxt = w[k + 1];
        r[k] = __funnelshift_r(cur, nxt, sh);
        cur = nxt;
    }
}

// Byte layout of one 64-token stage: code planes, then norm planes, of keys then
// values (each plane's rows contiguous).
template <int KO, int KN, int VO, int VN, bool KP = false>
struct MStage {
    static constexpr int R = kStageRows;
    static constexpr int kRKo = kDO * KO / 8, kRKn = kDN * KN / 8, kRVo = kDO * VO / 8, kRVn = kDN * VN / 8;
    static constexpr int kKOC = 0;
    static constexpr int kKNC = kKOC + R * kRKo;
    static constexpr int kKON = kKNC + R * kRKn;
    static constexpr int kKNN = kKON + R * 4;
    static constexpr int kVOC = kKNN + R * 4;
    static constexpr int kVNC = kVOC + R * kRVo;
    static constexpr int kVON = kVNC + R * kRVn;
    static constexpr int kVNN = kVON + R * 4;
    // prod keys: the parts' sign rows (32 and 96 signs) and residual norms
    static constexpr int kKOS = kVNN + R * 4;
    static constexpr int kKNS = kKOS + (KP ? R * 4 : 0);
    static constexpr int kKOR = kKNS + (KP ? R * 12 : 0);
    static constexpr int kKNR = kKOR + (KP ? R * 4 : 0);
    static constexpr int kBytes = kKNR + (KP ? R * 4 : 0);
    static constexpr int kRowBytes = kRKo + kRKn + kRVo + kRVn + 16 + (KP ? 24 : 0);
    static_assert(kRowBytes * R == kBytes, "stage layout");
    static_assert(kRKo % 4 == 0 && kRKn % 4 == 0 && kRVo % 4 == 0 && kRVn % 4 == 0, "code rows of whole words");
};

// Shared memory: four decode tables (each at a multiple of its power-of-two
// size), rotated and raw queries, the staging ring; then the combine and merge
// phases reuse the bytes.
template <int KO, int KN, int VO, int VN, bool KP = false>
struct MSmem {
    static constexpr int W = kMW;
    static constexpr int kThreads = (W + 1) * 32;
    static constexpr size_t kSz[4] = {Table<KO>::kBytes, Table<KN>::kBytes, Table<VO>::kBytes, Table<VN>::kBytes};
    static constexpr size_t kBig = 32768;
    static constexpr size_t kTabS = 0;  // the QJL sign table (prod keys, 32 KB) comes first
    static constexpr size_t kSgn = KP ? KSignTable::kBytes : 0;
    static_assert(KSignTable::kBytes == kBig, "sign table size");
    static constexpr size_t table_offset(int which) {  // the 32 KB tables first, then the others
        size_t off = kSgn;
        for (int pass = 0; pass < 2; ++pass)
            for (int i = 0; i < 4; ++i)
                if ((pass == 0) == (kSz[i] == kBig)) {
                    if (i == which) return off;
                    off += kSz[i];
                }
        return off;
    }
    static constexpr size_t kTabKO = table_offset(0), kTabKN = table_offset(1), kTabVO = table_offset(2),
                            kTabVN = table_offset(3);
    static constexpr size_t kQ = kSgn + kSz[0] + kSz[1] + kSz[2] + kSz[3];  // [kHeads][D] q′ (fp32)
    static constexpr size_t kQsc = kQ + (size_t)kHeads * D * 4;     // [kHeads]
    static constexpr size_t kQin = kQsc + kHeads * 4 + 16;          // [kHeads][D] raw q (query dtype)
    static constexpr size_t kQg = kQin + (size_t)kHeads * D * 4;    // [kHeads][D] permuted q (fp32)
    static constexpr size_t kPerm = kQg + (size_t)kHeads * D * 4;   // [D] perm_k
    static constexpr size_t kQ2 = kPerm + D * 4;                    // [kHeads][D] q″ (prod keys)
    static constexpr size_t kQsc2 = kQ2 + (KP ? (size_t)kHeads * D * 4 : 0);  // [kHeads]
    static constexpr size_t kStage = (kQsc2 + (KP ? kHeads * 4 : 0) + 127) & ~(size_t)127;
    static constexpr size_t kAlignSlack = kBig - 16;
    static constexpr size_t kLimit = 232448 - 2048;
    static constexpr int kStagesFit = (int)((kLimit - kAlignSlack - kStage) / MStage<KO, KN, VO, VN, KP>::kBytes);
    static constexpr int kStages = kStagesFit < kMaxStages ? kStagesFit : kMaxStages;
    static_assert(kStages >= 4, "too few staging stages fit in shared memory");
    static constexpr size_t kMain = kStage + (size_t)kStages * MStage<KO, KN, VO, VN, KP>::kBytes;
    // combine phase
    static constexpr size_t kWM = 0;
    static constexpr size_t kWL = kWM + W * kHeads * 4;
    static constexpr size_t kWF = kWL + W * kHeads * 4;
    static constexpr size_t kWO = kWF + W * kHeads * 4;
    static constexpr size_t kCombine = kWO + (size_t)W * kHeads * D * 4;
    // merge phase
    static constexpr int kMaxSplits = kMaxSplitsMerged;
    static constexpr size_t kMWt = 0;
    static constexpr size_t kML = kMWt + (size_t)kHeads * kMaxSplits * 4;
    static constexpr int kMRow = D + 8;
    static constexpr size_t kMO = (kML + kHeads * 4 + 15) & ~(size_t)15;
    static constexpr int kMC = 32;
    static constexpr size_t kMS = kMO + (size_t)kHeads * kMRow * 4;
    static constexpr size_t kMPerm = kMS + (size_t)kMC * kHeads * D * 4;  // [D] perm_v
    static constexpr size_t kMerge = kMPerm + D * 4;
    static_assert(kQin % 16 == 0 && kQg % 16 == 0 && kPerm % 16 == 0 && kMS % 16 == 0 && kMPerm % 16 == 0,
                  "16-byte aligned copy destinations");
    static constexpr size_t kBytes0 = kMain + kAlignSlack > kCombine ? kMain + kAlignSlack : kCombine;
    static constexpr size_t kBytes = kBytes0 > kMerge ? kBytes0 : kMerge;
};

// Dim of the frame held by element e of pair τ of lane-run c in the value
// accumulators (pairs 0–3 of a run are outlier dims, 4–15 the rest).
__host__ __device__ constexpr int mixed_vdim(int c, int tau, int e) {
    return tau < 4 ? 8 * c + 2 * tau + e : kDO + 24 * c + 2 * (tau - 4) + e;
}

// B operand of blockdiag(A_o, A_n) (row-major, A_o 32 × 32 and A_n 96 × 96, bf16
// hi and lo) for output rows i0 … i0 + 7: this lane's 16-byte pieces of row
// i0 + g, zero outside the row's diagonal block (hilo_b's layout).
__device__ __forceinline__ void blockdiag_b(const uint16_t* Ohi, const uint16_t* Olo, const uint16_t* Nhi,
                                            const uint16_t* Nlo, int i0, int g, int c, uint4 (&bh)[kKB / 2],
                                            uint4 (&bl)[kKB / 2]) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const int row = i0 + g;
#pragma unroll
    for (int p2 = 0; p2 < kKB / 2; ++p2) {
        const int col = 32 * p2 + 8 * c;  // columns col … col + 7 of the frame
        if (row < kDO && col < kDO) {
            const int q = (row * kDO + col) >> 3;
            bh[p2] = __ldg(reinterpret_cast<const uint4*>(Ohi) + q);
            bl[p2] = __ldg(reinterpret_cast<const uint4*>(Olo) + q);
        } else if (row >= kDO && col >= kDO) {
            const int q = ((row - kDO) * kDN + (col - kDO)) >> 3;
            bh[p2] = __ldg(reinterpret_cast<const uint4*>(Nhi) + q);
            bl[p2] = __ldg(reinterpret_cast<const uint4*>(Nlo) + q);
        } else {
            bh[p2] = z;
            bl[p2] = z;
        }
    }
}

// A channel index from a permutation entry: out-of-range entries read channel 0
// and are recorded in the status word.
__device__ __forceinline__ int channel(int v, int* status) {
    if ((unsigned)v < (unsigned)D) return v;
    atomicExch(status, TQ_STATUS_BAD_CHANNEL);
    return 0;
}

struct MixedAcc {
    float O[kMT][4];
    float M, Mt, l;
};

// QJL terms (KP): AS = [Q″_hi; Q″_lo] fragments, stab the lane's sign-table base,
// fSo, fSn the parts' score factors of the sign sums.
template <int KO, int KN, int VO, int VN, bool KP, bool FULL>
__device__ __forceinline__ void mixed_step(MixedAcc& st, const unsigned char* stp, int r0, int tb, int t1,
                                           const KDecoder<KO>& dko, const KDecoder<KN>& dkn, const Decoder<VO>& dvo,
                                           const Decoder<VN>& dvn, const uint32_t (&AQ)[kKB][4],
                                           const uint32_t (&AS)[KP ? kKB : 1][4], uint32_t stab, float fKo, float fKn,
                                           float fSo, float fSn, const MixedTcArgs& a, size_t head0, int G, int g,
                                           int c) {
    using ST = MStage<KO, KN, VO, VN, KP>;
    constexpr int NWKN = (24 * KN + 31) / 32;
    // ---- scores of head g, outlier part (k blocks 0–1) and the rest (2–7); with
    // prod keys the sign sums of the two parts as well
    float So[2][4], Sn[2][4], Qo[KP ? 2 : 1][4], Qn[KP ? 2 : 1][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
#pragma unroll
        for (int i = 0; i < 4; ++i) So[n][i] = Sn[n][i] = 0.f;
        if constexpr (KP) {
#pragma unroll
            for (int i = 0; i < 4; ++i) Qo[n][i] = Qn[n][i] = 0.f;
            // the lane's sign bytes: outlier byte c, then the rest's bytes 3c … 3c + 2
            const int row = r0 + 8 * n + g;
            uint32_t sw[1];
            lane_run<1, 24, 1>(stp + ST::kKNS + row * 12, c, sw);
            const uint32_t ws = (uint32_t)stp[ST::kKOS + row * 4 + c] | (sw[0] << 8);
#pragma unroll
            for (int j = 0; j < kKB / 2; ++j) {  // byte j: k blocks 2j, 2j + 1
                const uint4 f = lds128(field_off<8, 7>(&ws, 8 * j) | stab);
                float (&acc)[4] = j == 0 ? Qo[n] : Qn[n];
                mma16816(acc, AS[2 * j][0], AS[2 * j][1], AS[2 * j][2], AS[2 * j][3], f.x, f.y);
                mma16816(acc, AS[2 * j + 1][0], AS[2 * j + 1][1], AS[2 * j + 1][2], AS[2 * j + 1][3], f.z, f.w);
            }
        }
        const int row = r0 + 8 * n + g;
        uint32_t wo[1], wn[NWKN];
        lane_run<KO, 8, 1>(stp + ST::kKOC + row * ST::kRKo, c, wo);
        lane_run<KN, 24, NWKN>(stp + ST::kKNC + row * ST::kRKn, c, wn);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            uint32_t b0, b1;
            dko.frag(wo, kb, b0, b1);
            mma16816(So[n], AQ[kb][0], AQ[kb][1], AQ[kb][2], AQ[kb][3], b0, b1);
        }
        if constexpr (KN == 1) {
            // 1-bit codes are ±c₁: the ±1 sign table gives their fragments over the
            // run's contiguous dims (c₁ is folded into fKn)
            static_assert(!(KN == 1) || KP, "1-bit codes of the rest need the sign table");
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const uint4 f = lds128(field_off<8, 7>(wn, 8 * j) | stab);
                mma16816(Sn[n], AQ[2 + 2 * j][0], AQ[2 + 2 * j][1], AQ[2 + 2 * j][2], AQ[2 + 2 * j][3], f.x, f.y);
                mma16816(Sn[n], AQ[3 + 2 * j][0], AQ[3 + 2 * j][1], AQ[3 + 2 * j][2], AQ[3 + 2 * j][3], f.z, f.w);
            }
        } else {
#pragma unroll
            for (int kb = 2; kb < kKB; ++kb) {
                uint32_t b0, b1;
                dkn.frag(wn, kb - 2, b0, b1);
                mma16816(Sn[n], AQ[kb][0], AQ[kb][1], AQ[kb][2], AQ[kb][3], b0, b1);
            }
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
    float kno[4], knn[4], vno[4], vnn[4], kro[KP ? 4 : 1], krn[KP ? 4 : 1];
    norms(ST::kKON, kno);
    norms(ST::kKNN, knn);
    norms(ST::kVON, vno);
    norms(ST::kVNN, vnn);
    if constexpr (KP) {
        norms(ST::kKOR, kro);
        norms(ST::kKNR, krn);
    }
    // z = s·log2e + log2 max(‖v_o‖, ‖v_n‖), −∞ past the chunk
    // rows past the chunk may hold anything (whole stages are copied): their
    // exponents are −∞ and their norm ratios 0
    float z[4], lv[4], rv[4], ro[4], rn[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int n = i >> 1, j = i & 1;
        const bool live = FULL || tb + 8 * n + 2 * c + j < t1;
        const float vm = fmaxf(fmaxf(vno[i], vnn[i]), 1e-30f);
        lv[i] = lg2(vm);
        rv[i] = rcp(vm);
        ro[i] = live ? vno[i] * rv[i] : 0.f;  // ≤ 1
        rn[i] = live ? vnn[i] * rv[i] : 0.f;
        float s = fmaf(fKo * kno[i], So[n][j] + So[n][2 + j], fKn * knn[i] * (Sn[n][j] + Sn[n][2 + j]));
        if constexpr (KP) {
            s = fmaf(fSo * kno[i] * kro[i], Qo[n][j] + Qo[n][2 + j], s);
            s = fmaf(fSn * knn[i] * krn[i], Qn[n][j] + Qn[n][2 + j], s);
        }
        z[i] = live ? s + lv[i] : -INFINITY;
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
        const float corr = Mn == -INFINITY ? 1.f : ex2(st.M - Mn);
        st.M = Mn;
        st.Mt = Mn + kSlack;
        st.l *= corr;
        const float cA = __shfl_sync(0xffffffffu, corr, 8 * c), cB = __shfl_sync(0xffffffffu, corr, 8 * c + 4);
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
            st.O[m][0] *= cA;
            st.O[m][1] *= cB;
            st.O[m][2] *= cA;
            st.O[m][3] *= cB;
        }
    }
    float po[4], pn[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float p = ex2(z[i] - st.M);
        st.l = fmaf(p, rv[i], st.l);
        po[i] = p * ro[i];
        pn[i] = p * rn[i];
    }
    const uint32_t PO0 = pack_h2(po[0], po[1]), PO1 = pack_h2(po[2], po[3]);
    const uint32_t PN0 = pack_h2(pn[0], pn[1]), PN1 = pack_h2(pn[2], pn[3]);
    // ---- values: Oᵀ += Ṽᵀ·P′ᵀ, m tiles 0–1 outlier dims, 2–7 the rest
    {
        uint32_t oa[1], ob[1];
        constexpr int NWVN = (24 * VN + 31) / 32;
        uint32_t va[NWVN], vb[NWVN];
        lane_run<VO, 8, 1>(stp + ST::kVOC + (r0 + g) * ST::kRVo, c, oa);
        lane_run<VO, 8, 1>(stp + ST::kVOC + (r0 + g + 8) * ST::kRVo, c, ob);
        lane_run<VN, 24, NWVN>(stp + ST::kVNC + (r0 + g) * ST::kRVn, c, va);
        lane_run<VN, 24, NWVN>(stp + ST::kVNC + (r0 + g + 8) * ST::kRVn, c, vb);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            uint32_t x0, x1, y0, y1;
            dvo.pairs(oa, m, x0, x1);
            dvo.pairs(ob, m, y0, y1);
            mma16816(st.O[m], mov_trans(x0), mov_trans(x1), mov_trans(y0), mov_trans(y1), PO0, PO1);
        }
#pragma unroll
        for (int m = 2; m < kMT; ++m) {
            uint32_t x0, x1, y0, y1;
            dvn.pairs(va, m - 2, x0, x1);
            dvn.pairs(vb, m - 2, y0, y1);
            mma16816(st.O[m], mov_trans(x0), mov_trans(x1), mov_trans(y0), mov_trans(y1), PN0, PN1);
        }
    }
}

template <int KO, int KN, int VO, int VN, bool KP>
__device__ __forceinline__ void merge_mixed(const MixedTcArgs& a, unsigned char* smem, size_t head0, int G) {
    using SM = MSmem<KO, KN, VO, VN, KP>;
    constexpr int NT = SM::kThreads, NW = NT / 32, MR = SM::kMRow;
    float* wts = reinterpret_cast<float*>(smem + SM::kMWt);
    float* linv = reinterpret_cast<float*>(smem + SM::kML);
    float* mo = reinterpret_cast<float*>(smem + SM::kMO);
    int* pv = reinterpret_cast<int*>(smem + SM::kMPerm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int ns = a.n_splits;
    // out = blockdiag(Π_oᵀ, Π_nᵀ)·(acc/l), scattered to the channels by perm_v; the
    // matrix operands are loaded first
    constexpr int kJobs = D / 8, kPer = (kJobs + NW - 1) / NW;
    uint4 bh[kPer][kKB / 2], bl[kPer][kKB / 2];
#pragma unroll
    for (int u = 0; u < kPer; ++u)
        if (warp + u * NW < kJobs)
            blockdiag_b(a.vPiT_hi[0], a.vPiT_lo[0], a.vPiT_hi[1], a.vPiT_lo[1], 8 * (warp + u * NW), g, c, bh[u],
                        bl[u]);
    __shared__ __align__(8) uint64_t s_mbar;
    float* stg = reinterpret_cast<float*>(smem + SM::kMS);
    constexpr int kMC = SM::kMC;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&s_mbar, 1);
        sm100::fence_barrier_init();
    }
    if (threadIdx.x < D) pv[threadIdx.x] = channel(__ldg(a.perm_v + threadIdx.x), a.status);
    __syncthreads();
    auto stage_round = [&](int s0) {
        if (threadIdx.x == 0) {
            const uint32_t bytes = (uint32_t)min(kMC, ns - s0) * D * 4;
            asm volatile("fence.proxy.async;" ::: "memory");
            sm100::mbar_arrive_expect_tx(&s_mbar, G * bytes);
            for (int h = 0; h < G; ++h)
                bulk_g2s(smem_addr(stg + (size_t)h * kMC * D), a.pacc + ((head0 + h) * ns + s0) * D, bytes,
                         smem_addr(&s_mbar));
        }
    };
    stage_round(0);
    if (warp < G) {
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
    const int th = threadIdx.x / (D / 4), tj = threadIdx.x % (D / 4);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0, round = 0; s0 < ns; s0 += kMC, ++round) {
        const bool ok = sm100::mbar_wait(&s_mbar, (uint32_t)(round & 1), a.status, kDecodeMergeTimeout);
        __syncthreads();
        const int nsc = min(kMC, ns - s0);
        if (ok && th < G) {
            const float* w = wts + th * SM::kMaxSplits + s0;
            const float4* x = reinterpret_cast<const float4*>(stg) + (size_t)th * kMC * (D / 4) + tj;
            for (int sp = 0; sp < nsc; ++sp) {
                const float ws = w[sp];
                const float4 v = x[sp * (D / 4)];
                o = make_float4(fmaf(ws, v.x, o.x), fmaf(ws, v.y, o.y), fmaf(ws, v.z, o.z), fmaf(ws, v.w, o.w));
            }
        }
        if (s0 + kMC < ns) {
            __syncthreads();
            stage_round(s0 + kMC);
        }
    }
    if (th < kHeads) {
        const float li = th < G ? linv[th] : 0.f;
        *reinterpret_cast<float4*>(mo + th * MR + 4 * tj) = make_float4(o.x * li, o.y * li, o.z * li, o.w * li);
    }
    __syncthreads();
    uint32_t A[kKB][4];
    hilo_a(mo + g * MR, c, A);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int job = warp + u * NW;
        if (job >= kJobs) break;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        hilo_mma(acc, A, bh[u], bl[u]);
        if (g < G) {
            float* orow = a.out + (head0 + g) * D;
            orow[pv[8 * job + 2 * c]] = acc[0] + acc[2];
            orow[pv[8 * job + 2 * c + 1]] = acc[1] + acc[3];
        }
    }
}

template <int KO, int KN, int VO, int VN, bool KP>
__global__ void __launch_bounds__(MSmem<KO, KN, VO, VN, KP>::kThreads, 1)
    decode_mixed_mma_kernel(const __grid_constant__ MixedTcArgs a) {
    using SM = MSmem<KO, KN, VO, VN, KP>;
    using ST = MStage<KO, KN, VO, VN, KP>;
    constexpr int W = SM::W;
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sbase = smem_addr(smem);
    unsigned char* mp = smem + (((sbase + (uint32_t)SM::kBig - 1u) & ~((uint32_t)SM::kBig - 1u)) - sbase);
    float* qsh = reinterpret_cast<float*>(mp + SM::kQ);   // [kHeads][D] q′
    float* qsc = reinterpret_cast<float*>(mp + SM::kQsc);  // [kHeads]
    __shared__ int s_last;

    const int hb = blockIdx.y % a.n_hblocks, kvh = blockIdx.y / a.n_hblocks;
    const int G = min(kHeads, a.G - hb * kHeads);
    const int split = blockIdx.x, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int t0 = split * a.chunk;
    int t1 = t0, ntiles = 0, nstages = 0;
    // The kernel is the programmatic dependent of the ticket clearing kernel, so
    // the kernels before that one may still run: lengths, cache planes, queries,
    // permutations and tickets are read only after griddepcontrol.wait.
    auto read_length = [&]() {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int L = a.seq_lens[b];
        L = L < 0 ? 0 : (L > a.T_max ? a.T_max : L);
        t1 = min(t0 + a.chunk, L);
        ntiles = t1 > t0 ? (t1 - t0 + kTile - 1) / kTile : 0;
        nstages = (ntiles + kStageRows / kTile - 1) / (kStageRows / kTile);
    };
    const size_t head0 = (size_t)b * a.Hq + (size_t)kvh * a.G + (size_t)hb * kHeads;
    const int64_t rowbase = ((int64_t)b * a.Hkv + kvh) * a.T_max;

    // the matrices every CTA (Π_o, Π_n of the keys) or the merging CTAs (Π_oᵀ, Π_nᵀ
    // of the values) read: one L2 prefetch per 128-byte line over the grid
    {
        const int nct = gridDim.x * gridDim.y * gridDim.z;
        const int cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        constexpr int kLo = kDO * kDO * 2 / 128, kLn = kDN * kDN * 2 / 128, kPer = 2 * (kLo + kLn);
        const int l = cta + nct * (int)threadIdx.x;
        if (l < 2 * kPer) {
            const int side = l / kPer, r = l % kPer;  // keys, then values
            const int m = r < 2 * kLo ? r / kLo : 2 + (r - 2 * kLo) / kLn;
            const int line = r < 2 * kLo ? r % kLo : (r - 2 * kLo) % kLn;
            const uint16_t* const* mats = side == 0 ? a.kPi_hi : a.vPiT_hi;
            const uint16_t* const* matl = side == 0 ? a.kPi_lo : a.vPiT_lo;
            const uint16_t* base = (m & 1) ? matl[m >> 1] : mats[m >> 1];
            asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(base + 64 * line));
        }
    }

    const uint8_t* kco = a.kc[0] + (size_t)rowbase * ST::kRKo;
    const uint8_t* kcn = a.kc[1] + (size_t)rowbase * ST::kRKn;
    const float* kno = a.kn[0] + rowbase;
    const float* knn = a.kn[1] + rowbase;
    const uint8_t* vco = a.vc[0] + (size_t)rowbase * ST::kRVo;
    const uint8_t* vcn = a.vc[1] + (size_t)rowbase * ST::kRVn;
    const float* vno = a.vn[0] + rowbase;
    const float* vnn = a.vn[1] + rowbase;
    const uint8_t* kso = KP ? a.ks[0] + (size_t)rowbase * 4 : nullptr;
    const uint8_t* ksn = KP ? a.ks[1] + (size_t)rowbase * 12 : nullptr;
    const float* kro = KP ? a.kr[0] + rowbase : nullptr;
    const float* krn = KP ? a.kr[1] + rowbase : nullptr;

    const uint32_t ring = smem_addr(mp + SM::kStage);
    __shared__ __align__(8) uint64_t s_full[SM::kStages], s_empty[SM::kStages];
    const bool producer = warp == W;
    // one bulk copy per plane and stage (T_max % 4 == 0: every copy 16-byte sized and aligned)
    auto produce = [&](int i) {
        const int tb = t0 + i * kStageRows;
        const uint32_t dst = ring + (uint32_t)((i % SM::kStages) * ST::kBytes);
        const uint32_t bar = smem_addr(&s_full[i % SM::kStages]);
        const uint32_t rows = (uint32_t)min(kStageRows, a.T_max - tb);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(rows * ST::kRowBytes)
                     : "memory");
        bulk_g2s(dst + ST::kKOC, kco + (size_t)tb * ST::kRKo, rows * ST::kRKo, bar);
        bulk_g2s(dst + ST::kKNC, kcn + (size_t)tb * ST::kRKn, rows * ST::kRKn, bar);
        bulk_g2s(dst + ST::kKON, kno + tb, rows * 4, bar);
        bulk_g2s(dst + ST::kKNN, knn + tb, rows * 4, bar);
        bulk_g2s(dst + ST::kVOC, vco + (size_t)tb * ST::kRVo, rows * ST::kRVo, bar);
        bulk_g2s(dst + ST::kVNC, vcn + (size_t)tb * ST::kRVn, rows * ST::kRVn, bar);
        bulk_g2s(dst + ST::kVON, vno + tb, rows * 4, bar);
        bulk_g2s(dst + ST::kVNN, vnn + tb, rows * 4, bar);
        if constexpr (KP) {
            bulk_g2s(dst + ST::kKOS, kso + (size_t)tb * 4, rows * 4, bar);
            bulk_g2s(dst + ST::kKNS, ksn + (size_t)tb * 12, rows * 12, bar);
            bulk_g2s(dst + ST::kKOR, kro + tb, rows * 4, bar);
            bulk_g2s(dst + ST::kKNR, krn + tb, rows * 4, bar);
        }
    };
    if (producer && lane == 0) {
        for (int i = 0; i < SM::kStages; ++i) {
            sm100::mbar_init(&s_full[i], 1);
            sm100::mbar_init(&s_empty[i], kStageRows / kTile);
        }
        sm100::fence_barrier_init();
    }
    __syncthreads();
    auto consumers_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(W * 32) : "memory"); };

    MixedAcc st;
#pragma unroll
    for (int m = 0; m < kMT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) st.O[m][i] = 0.f;
    st.M = -INFINITY;
    st.Mt = -INFINITY;
    st.l = 0.f;

    if (producer) {
        read_length();
        if (lane == 0)
            for (int i = 0; i < min(nstages, SM::kStages); ++i) produce(i);
        for (int i = SM::kStages; i < nstages; ++i) {
            const bool ok = sm100::mbar_wait(&s_empty[i % SM::kStages], (uint32_t)((i / SM::kStages - 1) & 1), a.status,
                                             kDecodeStageTimeout);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) produce(i);
        }
    } else {
        // ---- prologue (consumer warps): tables, q gathered by perm_k, q′, scales
        constexpr int NC = W * 32;
        constexpr int kJobs = D / 8, kPer = (kJobs + W - 1) / W;
        uint4 bh[kPer][kKB / 2], bl[kPer][kKB / 2];
#pragma unroll
        for (int u = 0; u < kPer; ++u)
            if (warp + u * W < kJobs)
                blockdiag_b(a.kPi_hi[0], a.kPi_lo[0], a.kPi_hi[1], a.kPi_lo[1], 8 * (warp + u * W), g, c, bh[u],
                            bl[u]);
        unsigned char* qin = mp + SM::kQin;
        int* pk = reinterpret_cast<int*>(mp + SM::kPerm);
        Table<KO>::fill(mp + SM::kTabKO, a.kcb[0], threadIdx.x, NC);
        Table<KN>::fill(mp + SM::kTabKN, a.kcb[1], threadIdx.x, NC);
        Table<VO>::fill(mp + SM::kTabVO, a.vcb[0], threadIdx.x, NC);
        Table<VN>::fill(mp + SM::kTabVN, a.vcb[1], threadIdx.x, NC);
        if constexpr (KP) KSignTable::fill(mp + SM::kTabS, threadIdx.x, NC);
        asm volatile("griddepcontrol.wait;" ::: "memory");
        {
            const int rowq = a.q_f32 ? D / 4 : D / 8;
            const unsigned char* qb = static_cast<const unsigned char*>(a.q) + head0 * D * (a.q_f32 ? 4 : 2);
            for (int idx = threadIdx.x; idx < kHeads * rowq; idx += NC) {
                const bool live = idx / rowq < G;
                cp_async16(smem_addr(qin) + 16u * (uint32_t)idx, live ? qb + 16 * idx : qb, live ? 16u : 0u);
            }
            for (int idx = threadIdx.x; idx < D / 4; idx += NC)
                cp_async16(smem_addr(pk) + 16u * (uint32_t)idx, a.perm_k + 4 * idx, 16u);
            cp_async_commit();
        }
        cp_async_wait<0>();
        consumers_sync();
        // q gathered into the frame's channel order: qg[h][i] = q[h][perm_k[i]]
        float* qg = reinterpret_cast<float*>(mp + SM::kQg);
        for (int idx = threadIdx.x; idx < kHeads * D; idx += NC) {
            const int h = idx / D, i = idx % D;
            const int ch = channel(pk[i], a.status);
            qg[idx] = a.q_f32 ? reinterpret_cast<const float*>(qin)[h * D + ch]
                              : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(qin)[h * D + ch]);
        }
        consumers_sync();
        {
            uint32_t A[kKB][4];
            hilo_a(qg + g * D, c, A);
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int job = warp + u * W;
                if (job < kJobs) {
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    hilo_mma(acc, A, bh[u], bl[u]);
                    qsh[g * D + 8 * job + 2 * c] = acc[0] + acc[2];
                    qsh[g * D + 8 * job + 2 * c + 1] = acc[1] + acc[3];
                }
            }
            if constexpr (KP) {  // q″ = blockdiag(S_o, S_n)·(P q), the same way
                float* qsh2 = reinterpret_cast<float*>(mp + SM::kQ2);
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const int job = warp + u * W;
                    if (job < kJobs) {
                        uint4 sh[kKB / 2], sl[kKB / 2];
                        blockdiag_b(a.kS_hi[0], a.kS_lo[0], a.kS_hi[1], a.kS_lo[1], 8 * job, g, c, sh, sl);
                        float acc[4] = {0.f, 0.f, 0.f, 0.f};
                        hilo_mma(acc, A, sh, sl);
                        qsh2[g * D + 8 * job + 2 * c] = acc[0] + acc[2];
                        qsh2[g * D + 8 * job + 2 * c + 1] = acc[1] + acc[3];
                    }
                }
            }
        }
        consumers_sync();
        for (int h = warp; h < kHeads; h += W) {
            float m1 = 0.f, m2 = 0.f;
            for (int j = lane; j < D; j += 32) {
                m1 = fmaxf(m1, fabsf(qsh[h * D + j]));
                if constexpr (KP) m2 = fmaxf(m2, fabsf(reinterpret_cast<const float*>(mp + SM::kQ2)[h * D + j]));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
                m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
            }
            if (lane == 0) {
                qsc[h] = m1 > 0.f ? m1 : 1.f;
                if constexpr (KP) reinterpret_cast<float*>(mp + SM::kQsc2)[h] = m2 > 0.f ? m2 : 1.f;
            }
        }
        consumers_sync();
        read_length();
        // A fragments of head g: this lane's dims 8c … 8c + 7 and 32 + 24c … 32 + 24c + 23
        uint32_t AQ[kKB][4];
        {
            const float i1 = 1.f / qsc[g];
            float q1[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) q1[k] = qsh[g * D + 8 * c + k];
#pragma unroll
            for (int k = 0; k < 24; ++k) q1[8 + k] = qsh[g * D + kDO + 24 * c + k];
#pragma unroll
            for (int kb = 0; kb < kKB; ++kb)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float x0 = q1[4 * kb + 2 * h] * i1, x1 = q1[4 * kb + 2 * h + 1] * i1;
                    const __half2 hh = __floats2half2_rn(x0, x1);
                    const float2 hf = __half22float2(hh);
                    AQ[kb][2 * h] = *reinterpret_cast<const uint32_t*>(&hh);
                    AQ[kb][2 * h + 1] = pack_h2(x0 - hf.x, x1 - hf.y);
                }
        }
        // [Q″_hi; Q″_lo] fragments of head g over the same dims (prod keys)
        uint32_t AS[KP ? kKB : 1][4];
        float fSo = 0.f, fSn = 0.f;
        const float scale2 = a.scale * kLog2e;
        if constexpr (KP) {
            const float* qsh2 = reinterpret_cast<const float*>(mp + SM::kQ2);
            const float qs2 = reinterpret_cast<const float*>(mp + SM::kQsc2)[g], i2 = 1.f / qs2;
            float q2[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) q2[k] = qsh2[g * D + 8 * c + k];
#pragma unroll
            for (int k = 0; k < 24; ++k) q2[8 + k] = qsh2[g * D + kDO + 24 * c + k];
#pragma unroll
            for (int kb = 0; kb < kKB; ++kb)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float x0 = q2[4 * kb + 2 * h] * i2, x1 = q2[4 * kb + 2 * h + 1] * i2;
                    const __half2 hh = __floats2half2_rn(x0, x1);
                    const float2 hf = __half22float2(hh);
                    AS[kb][2 * h] = *reinterpret_cast<const uint32_t*>(&hh);
                    AS[kb][2 * h + 1] = pack_h2(x0 - hf.x, x1 - hf.y);
                }
            fSo = scale2 * a.kgamma[0] * qs2;
            fSn = scale2 * a.kgamma[1] * qs2;
        }
        const uint32_t stab = KP ? KSignTable::lane_base(mp + SM::kTabS, lane) : 0u;
        static_assert(KO >= 2, "outlier codes of at least two bits");
        const float fKo = scale2 * qsc[g] / a.kcb[0].lut_scale;
        // 1-bit codes of the rest go through the ±1 sign table: scale by c₁
        const float fKn = KN == 1 ? scale2 * qsc[g] * a.kcb[1].c[1] : scale2 * qsc[g] / a.kcb[1].lut_scale;
        KDecoder<KO> dko;
        KDecoder<KN> dkn;
        Decoder<VO> dvo;
        Decoder<VN> dvn;
        dko.init(a.kcb[0], mp + SM::kTabKO, lane);
        dkn.init(a.kcb[1], mp + SM::kTabKN, lane);
        dvo.init(a.vcb[0], mp + SM::kTabVO, lane);
        dvn.init(a.vcb[1], mp + SM::kTabVN, lane);
        for (int tile = warp; tile < ntiles; tile += W) {
            constexpr int kTilesPerStage = kStageRows / kTile;
            const int stage = tile / kTilesPerStage, slot = stage % SM::kStages;
            const bool ok = sm100::mbar_wait(&s_full[slot], (uint32_t)((stage / SM::kStages) & 1), a.status,
                                             kDecodeStageTimeout);
            if (!__all_sync(0xffffffffu, ok)) break;
            const int tb = t0 + tile * kTile, r0 = (tile % kTilesPerStage) * kTile;
            const unsigned char* stp = mp + SM::kStage + (size_t)slot * ST::kBytes;
            if (tb + kTile <= t1)
                mixed_step<KO, KN, VO, VN, KP, true>(st, stp, r0, tb, t1, dko, dkn, dvo, dvn, AQ, AS, stab, fKo, fKn,
                                                     fSo, fSn, a, head0, G, g, c);
            else
                mixed_step<KO, KN, VO, VN, KP, false>(st, stp, r0, tb, t1, dko, dkn, dvo, dvn, AQ, AS, stab, fKo,
                                                      fKn, fSo, fSn, a, head0, G, g, c);
            __syncwarp();
            if (lane == 0) sm100::mbar_arrive(&s_empty[slot]);
        }
    }

    // ---- combine the warps of this CTA into one split partial per head
    st.l += __shfl_xor_sync(0xffffffffu, st.l, 1);
    st.l += __shfl_xor_sync(0xffffffffu, st.l, 2);
    __syncthreads();
    float* wM = reinterpret_cast<float*>(smem + SM::kWM);
    float* wL = reinterpret_cast<float*>(smem + SM::kWL);
    float* wF = reinterpret_cast<float*>(smem + SM::kWF);
    float* wO = reinterpret_cast<float*>(smem + SM::kWO);
    constexpr int kFrag = kMT * 4 * 32;
    if (!producer) {
        if (c == 0) {
            wM[warp * kHeads + g] = st.M;
            wL[warp * kHeads + g] = st.l;
        }
#pragma unroll
        for (int m = 0; m < kMT; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) wO[warp * kFrag + (m * 4 + i) * 32 + lane] = st.O[m][i];
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
    // element (m, i, lane): head 2c + (i & 1); row g (i < 2) or g + 8 of m tile m is
    // element g & 1 of pair 2m + (i >> 1) of run g >> 1; the outlier tiles carry
    // the outlier codebook's table scale, the others the rest's
    const float inv_o = 1.f / a.vcb[0].lut_scale, inv_n = 1.f / a.vcb[1].lut_scale;
    for (int f = threadIdx.x; f < kFrag; f += blockDim.x) {
        const int fl = f & 31, fi = (f >> 5) & 3, fm = f >> 7;
        const int h = 2 * (fl & 3) + (fi & 1), fg = fl >> 2;
        if (h >= G) continue;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) o = fmaf(wF[w * kHeads + h], wO[w * kFrag + f], o);
        const size_t ps = (head0 + h) * a.n_splits + split;
        a.pacc[ps * D + mixed_vdim(fg >> 1, 2 * fm + (fi >> 1), fg & 1)] = o * (fm < 2 ? inv_o : inv_n);
    }

    __syncthreads();
    if (threadIdx.x == 0) {
        const int group = (b * a.Hkv + kvh) * a.n_hblocks + hb;
        int old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(a.cnt + group) : "memory");
        s_last = old == a.n_splits - 1;
    }
    __syncthreads();
    if (!s_last) return;
    merge_mixed<KO, KN, VO, VN, KP>(a, smem, head0, G);
}

template <int KO, int KN, int VO, int VN, bool KP>
int launch_mixed_tc(const MixedTcArgs& a, dim3 grid, cudaStream_t s) {
    using SM = MSmem<KO, KN, VO, VN, KP>;
    static_assert(SM::kBytes <= 232448 - 1024, "mixed decode shared memory above the per-CTA limit");
    auto fn = decode_mixed_mma_kernel<KO, KN, VO, VN, KP>;
    static std::atomic<uint64_t> smem_set{0};
    const int rc = ensure_smem_attr(smem_set, (const void*)fn, (int)SM::kBytes, "mixed decode smem attribute");
    if (rc != TQ_OK) return rc;
    // the programmatic dependent of the ticket clearing kernel launched before it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(SM::kThreads);
    cfg.dynamicSmemBytes = SM::kBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, a);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "mixed decode (tensor-core) launch");
}

}  // namespace
}  // namespace mmadec

// code bits (b_o, b_n) of keys and values: the instantiated combinations
bool mixed_tc_bits_supported(int ko, int kn, int vo, int vn, bool kp) {
    auto ok = [](int o, int n) { return (o == 3 && n == 2) || (o == 4 && n == 3) || (o == 4 && n == 2); };
    if (kp) return ok(ko + 1, kn + 1) && vo == ko + 1 && vn == kn + 1;
    return ok(ko, kn) && ko == vo && kn == vn;
}

int launch_mixed_decode_tc(const MixedTcArgs& a, dim3 grid, int ko, int kn, cudaStream_t s) {
    using namespace mmadec;
    if (a.kp) {
        if (ko == 2 && kn == 1) return launch_mixed_tc<2, 1, 3, 2, true>(a, grid, s);
        if (ko == 3 && kn == 2) return launch_mixed_tc<3, 2, 4, 3, true>(a, grid, s);
        if (ko == 3 && kn == 1) return launch_mixed_tc<3, 1, 4, 2, true>(a, grid, s);
    } else {
        if (ko == 3 && kn == 2) return launch_mixed_tc<3, 2, 3, 2, false>(a, grid, s);
        if (ko == 4 && kn == 3) return launch_mixed_tc<4, 3, 4, 3, false>(a, grid, s);
        if (ko == 4 && kn == 2) return launch_mixed_tc<4, 2, 4, 2, false>(a, grid, s);
    }
    return fail(TQ_EUNSUPPORTED, "tensor-core mixed decode: bits (%d, %d)", ko, kn);
}

}  // namespace tq
