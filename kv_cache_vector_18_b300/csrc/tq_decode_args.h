// Arguments of the split-K decode kernels (CUDA-core and tensor-core), shared
// by tq_decode.cu and the tensor-core instantiation files.
#pragma once

#include "tq_internal.h"

namespace tq {

// Device pointers and shapes one split launch needs (see include/tq.h).
struct SplitArgs {
    const uint8_t* kcodes;
    const uint8_t* ksigns;
    const float* knorm;
    const float* krnorm;
    const uint8_t* vcodes;
    const uint8_t* vsigns;
    const float* vnorm;
    const float* vrnorm;
    const int32_t* seq_lens;
    const float* qr;
    const float* qs;
    float* pm;
    float* pl;
    float* pacc;
    float* pacc2;
    float* scores;
    Codebook kcb, vcb;
    int kb, vb;  // b_m of keys / values
    float kgamma, vgamma, scale;
    int B, Hq, Hkv, T_max, G, n_splits, chunk, n_hblocks;
    // Fused merge (tensor-core path): one ticket counter per (batch, KV head,
    // head block), zeroed before the launch (by the ticket clearing kernel, or by
    // the decode-step append);
    // the last split CTA of a group combines the partials and writes
    // out = Π_vᵀ·acc/l (+ S_vᵀ·acc2/l).
    int* cnt;
    const float* vPi;  // Π_v row-major [d][d]
    const float* vS;   // S_v row-major [d][d] (prod values)
    // Π_vᵀ = hi + lo and S_vᵀ = hi + lo, bf16 row-major [i][j]: the merge's matrix operands
    const uint16_t* vPiT_hi;
    const uint16_t* vPiT_lo;
    const uint16_t* vST_hi;
    const uint16_t* vST_lo;
    float* out;        // [B, Hq, d]
    // Query rotation inside the split kernel (tensor-core path): q′ = Π_k·q, q″ = S_k·q.
    const void* q;     // [B, Hq, d], bf16 or f32
    int q_f32;
    // 1: launched as the programmatic dependent of the decode-step append, which
    // writes neither q nor any cache row below the length it starts from (it
    // writes row seq_lens[b] of each slab, then bumps the lengths): q and those
    // rows may be read before griddepcontrol.wait.  0: nothing before it.
    int after_append;
    // the rotation on the tensor cores: Π_k = hi + lo, S_k = hi + lo, bf16 row-major [j][i]
    const uint16_t* kPi_hi;
    const uint16_t* kPi_lo;
    const uint16_t* kS_hi;
    const uint16_t* kS_lo;
    // the key handle's device status word: a staging wait that gives up records
    // kDecodeStageTimeout there
    int* status;
};

namespace mmadec {
// Tensor-core split kernel for d = 128, keys (kb, kprod) fixed per instantiation
// file, values dispatched at run time.  Heads are processed 8 per CTA.
constexpr int kHeadsPerCta = 8;
constexpr int D128 = 128;
constexpr int kMaxSplitsMerged = 256;  // splits the last CTA of a group can merge
constexpr int kDecodeStageTimeout = 30;  // status code of an expired tile-staging wait
constexpr int kDecodeMergeTimeout = 31;  // status code of an expired wait for the split partials
// resident split CTAs per SM of the tensor-core decode kernel (one 16- or 8-warp CTA)
constexpr int ctas_per_sm(bool /*vprod*/) { return 1; }
template <int KB, bool KP>
int launch_for_k(const SplitArgs& a, dim3 grid, int vb, bool vp, bool pdl, cudaStream_t s);
}  // namespace mmadec

}  // namespace tq
