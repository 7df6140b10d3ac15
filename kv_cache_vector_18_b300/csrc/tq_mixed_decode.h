// Arguments of the tensor-core mixed-precision decode (tq_decode_mixed_mma.cu):
// keys and values each split into an outlier part (index 0: 32 channels) and the
// rest (index 1: 96 channels) of d = 128; value parts mse quantizers, key parts
// both mse or both prod (kp).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "tq_internal.h"

namespace tq {

struct MixedTcArgs {
    const uint8_t* kc[2];  // code planes, rows ordered [B][Hkv][T_max]
    const float* kn[2];    // norm planes
    const uint8_t* vc[2];
    const float* vn[2];
    const int32_t* seq_lens;
    const int32_t* perm_k;  // [128]: the frame's channel i is perm_k[i]
    const int32_t* perm_v;
    float* pm;    // [B·Hq][n_splits] split maxima (natural-log units)
    float* pl;    // [B·Hq][n_splits] split sums
    float* pacc;  // [B·Hq][n_splits][128] split value sums in the value frame
    int* cnt;     // [B·Hq] merge tickets, zero on entry
    float* out;
    float* scores;
    Codebook kcb[2], vcb[2];
    float scale;
    int B, Hq, Hkv, T_max, G, n_splits, chunk, n_hblocks;
    const void* q;
    int q_f32;
    // Π of the key parts (bf16 hi/lo, row-major, 32 × 32 and 96 × 96) and Πᵀ of the value parts
    const uint16_t* kPi_hi[2];
    const uint16_t* kPi_lo[2];
    const uint16_t* vPiT_hi[2];
    const uint16_t* vPiT_lo[2];
    int* status;  // the outlier key handle's status word
    // prod key parts: QJL sign planes (4 and 12 bytes per row), residual norms,
    // S of each part (bf16 hi/lo, row-major) and √(π/2)/d_p
    int kp;
    const uint8_t* ks[2];
    const float* kr[2];
    const uint16_t* kS_hi[2];
    const uint16_t* kS_lo[2];
    float kgamma[2];
};

// The code bits (b_o, b_n) of the key and value parts with a tensor-core kernel:
// mse keys (3, 2), (4, 3), (4, 2) with values alike; prod keys (codes (2, 1),
// (3, 2), (3, 1), i.e. 3/2, 4/3, 4/2 bits with the sign) with mse values of the
// keys' total bits.
bool mixed_tc_bits_supported(int ko, int kn, int vo, int vn, bool kp);
int launch_mixed_decode_tc(const MixedTcArgs& a, dim3 grid, int ko, int kn, cudaStream_t s);

}  // namespace tq
