// Device helpers shared by the libtq kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq_internal.h"

namespace tq {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float load_elem(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_elem(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// Index of rotated coordinate y against the scaled boundaries: #{k : n·t_k < y}.
__device__ __forceinline__ int bucket_count(const Codebook& cb, float n, float y) {
    int c = 0;
#pragma unroll
    for (int k = 0; k < kMaxLevels - 1; ++k)
        if (k < cb.levels - 1) c += (n * cb.t[k] < y) ? 1 : 0;
    return c;
}

// Channels of one part of an outlier-channel split: element j of the part is
// channel ch[j] of a full row of d_full elements (ch == nullptr: channel j, the
// plain single-part row).  An index outside [0, d_full) is never dereferenced: it
// maps to channel 0 and records TQ_STATUS_BAD_CHANNEL.
struct ChannelMap {
    const int32_t* ch = nullptr;
    int d_full = 0;
    int* status = nullptr;
};

__device__ __forceinline__ int channel_of(const ChannelMap& cm, int j) {
    if (cm.ch == nullptr) return j;
    const int c = cm.ch[j];
    if ((unsigned)c < (unsigned)cm.d_full) return c;
    atomicExch(cm.status, TQ_STATUS_BAD_CHANNEL);
    return 0;
}

// Read code j (b bits, LSB-first bitstream) from a row held as 32-bit words.
__device__ __forceinline__ int read_code(const uint32_t* w, int j, int b) {
    int bit = j * b;
    int wi = bit >> 5, sh = bit & 31;
    uint32_t v = w[wi] >> sh;
    if (sh + b > 32) v |= w[wi + 1] << (32 - sh);
    return (int)(v & ((1u << b) - 1u));
}

}  // namespace tq
