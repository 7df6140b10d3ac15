// Internal declarations shared by the host API and the CUDA kernels of libtq.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <string>
#include <vector>

#include "tq.h"

namespace tq {

constexpr int kMaxLevels = 16;   // 2^b_m with b_m <= 4
constexpr int kMinD = 32;
constexpr int kMaxD = 256;
constexpr int kMaxGroup = 16;    // query heads per KV head

// Codebook passed by value to kernels (lives in the kernel-parameter bank).
struct Codebook {
    float c[kMaxLevels];       // centroids, unit-sphere scale, ascending
    float t[kMaxLevels - 1];   // decision boundaries (midpoints), ascending
    int levels;                // 2^b_m
    float lut_scale;           // σ ∈ [1, 2): f16(σ·c_k) is within ~1e-4 relative of σ·c_k for every k
};

// Float64 parameters of one quantizer, as built on the host.
struct HostParams {
    int d = 0, bits = 0, variant = 0, b_mse = 0, levels = 0;
    int rotation = 0;               // TQ_ROT_QR or TQ_ROT_HADAMARD
    uint64_t seed = 0;
    std::vector<double> Pi;         // [d*d] row-major, y = Pi x
    std::vector<double> S;          // [d*d] row-major (prod)
    std::vector<double> centroids;  // [levels]
    std::vector<double> bounds;     // [levels-1]
};

// Device copies of the matrices in the layouts each kernel reads.
struct DeviceParams {
    float* Pi = nullptr;    // [d*d]  Pi[j*d+i] = Π_ji   (column reads over i)
    float* PiT = nullptr;   // [d*d]  PiT[i*d+j] = Π_ji  (row reads over j)
    float* S = nullptr;     // [d*d]  S[j*d+i] = S_ji    (prod)
    float* ST = nullptr;    // [d*d]  ST[i*d+j] = S_ji   (prod)
    float* TT = nullptr;    // [d*d]  TT[j*d+i] = (S Πᵀ)_ij  (prod)
    // Tensor-core operands: Π = Π_hi + Π_lo as two bf16 matrices, row-major [j][i].
    uint16_t* Pi_hi = nullptr;
    uint16_t* Pi_lo = nullptr;
    uint16_t* S_hi = nullptr;  // S = S_hi + S_lo, bf16 row-major [j][i] (prod)
    uint16_t* S_lo = nullptr;
    // Πᵀ and Sᵀ split the same way, row-major [i][j] (the decode merge's x = Πᵀ·y)
    uint16_t* PiT_hi = nullptr;
    uint16_t* PiT_lo = nullptr;
    uint16_t* ST_hi = nullptr;  // (prod)
    uint16_t* ST_lo = nullptr;
    CUtensorMap tm_pi_hi;   // TMA maps over Pi_hi / Pi_lo, box {64, d}, 128-byte swizzle
    CUtensorMap tm_pi_lo;
    // Hadamard rotation: √d·Π = H·diag(σ) has entries ±1, exact in bf16, so the
    // quantize contraction takes it in one pass and scales the norm by 1/√d.
    uint16_t* Pm = nullptr;
    CUtensorMap tm_pm;
    // prod: T = S·Πᵀ = T_hi + T_lo as two f16 matrices, row-major [i][j], and TMA maps
    uint16_t* T_hi = nullptr;
    uint16_t* T_lo = nullptr;
    CUtensorMap tm_t_hi;
    CUtensorMap tm_t_lo;
    int* status = nullptr;  // device word: 0, or the code of a bounded wait that expired
    // device word after the status word: blocks of a decode-step append that have
    // finished (the last one resets it to 0)
    int* append_done = nullptr;
};

}  // namespace tq

struct tq_ctx {
    tq::HostParams hp;
    tq::DeviceParams dp;
    tq::Codebook cb;
    int device = 0;
    int num_sms = 0;
    int code_bytes = 0;
    int sign_bytes = 0;
    float gamma = 0.f;  // √(π/2)/d
    // rotation operand of the tensor-core quantize kernels: 2 passes (Π_hi, Π_lo) with
    // norm scale 1, or 1 pass over the ±1 Hadamard matrix with norm scale 1/√d
    int rot_passes = 2;
    float rot_norm_scale = 1.f;
};

namespace tq {

// Error reporting (thread-local message, returns the code for chaining).
int fail(int code, const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);
int check_device_ptr(const void* p, const char* name, bool required);

// Raise a kernel's dynamic shared-memory limit on the current device once (the
// attribute persists for the process).  `done` is the caller's per-kernel
// bitmask of device ordinals already configured.
inline int ensure_smem_attr(std::atomic<uint64_t>& done, const void* fn, int bytes, const char* what) {
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_relaxed) & bit) return TQ_OK;
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return cuda_fail(e, what);
    done.fetch_or(bit, std::memory_order_relaxed);
    return TQ_OK;
}

// Host parameter construction (tq_params.cpp).
int build_host_params(int d, int bits, int variant, int rotation, uint64_t seed, HostParams* out);

// 2-D bf16 TMA map: `inner` contiguous elements per row, `outer` rows `row_stride_bytes` apart,
// box {box_inner, box_outer}, 128-byte swizzle, out-of-range elements read as zero.
int encode_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);
// The same for an f16 matrix.
int encode_tmap_f16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                       uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

// Kernel launchers (one per .cu file).  Arguments are validated by the caller.
bool quantize_tc_supported(const tq_ctx& h, int x_dtype, int64_t n_rows);
int launch_expire_wait(const tq_ctx& h, int code, uint64_t limit_ns, cudaStream_t s);
// Outlier-channel mixed precision (tq_quantize.cu, tq_dequantize.cu, tq_mixed.cu):
// one part of a channel split quantized from / dequantized to full rows of d_full.
int launch_quantize_part(const tq_ctx& h, const void* x, int x_dtype, int64_t n_rows, int64_t stride,
                         const int32_t* ch, int d_full, const tq_planes& out, cudaStream_t s);
int launch_dequantize_part(const tq_ctx& h, const tq_planes& in, int64_t n_rows, const int32_t* ch, int d_full,
                           void* y, int y_dtype, cudaStream_t s);
// Tensor-core mixed quantize (tq_mixed_tc.cu): bf16 rows, mse parts, d = 128,
// d_o ∈ {32, 64}; scratch holds the combined rotation operand (hi and lo).
size_t mixed_tc_scratch_bytes();
bool mixed_quantize_tc_supported(const tq_ctx& ho, const tq_ctx& hn, int x_dtype, int64_t n_rows, int64_t stride,
                                 const void* scratch, size_t scratch_bytes);
int launch_mixed_quantize_tc(const tq_ctx& ho, const tq_ctx& hn, const int32_t* perm, const void* x, int64_t n_rows,
                             int64_t stride, const tq_planes& out_o, const tq_planes& out_n, void* scratch,
                             cudaStream_t s);
// Keys and values in one launch (both sides supported alone, the same d_o and
// bits, scratch of two operands: keys' first, values' second).
bool mixed_quantize_pair_tc_supported(const tq_ctx& hko, const tq_ctx& hkn, const tq_ctx& hvo, const tq_ctx& hvn,
                                      int x_dtype, int64_t k_rows, int64_t k_stride, int64_t v_rows,
                                      int64_t v_stride, const void* scratch, size_t scratch_bytes);
int launch_mixed_quantize_pair_tc(const tq_ctx& hko, const tq_ctx& hkn, const tq_ctx& hvo, const tq_ctx& hvn,
                                  const int32_t* perm_k, const int32_t* perm_v, const void* k, const void* v,
                                  int64_t k_rows, int64_t k_stride, int64_t v_rows, int64_t v_stride,
                                  const tq_planes& k_out_o, const tq_planes& k_out_n, const tq_planes& v_out_o,
                                  const tq_planes& v_out_n, void* scratch, cudaStream_t s);
struct MixedShape {
    int B = 0, Hq = 0, Hkv = 0, T_max = 0, d = 0, G = 0, n_splits = 1, chunk = 64;
    bool tc = false;  // the tensor-core mixed decode (tq_decode_mixed_mma.cu) runs it
};
struct MixedDecode {
    const tq_ctx* hk[2];  // key parts: outlier channels, the rest
    const tq_ctx* hv[2];
    const int32_t* perm_k;
    const int32_t* perm_v;
    const void* q;
    int q_dtype;
    tq_planes kc[2], vc[2];
    const int32_t* seq_lens;
    float scale;
    float* out;
    float* scores;
    void* workspace;
};
int mixed_plan(int d, int sms, bool vprod, bool tc, int B, int Hq, int Hkv, int T_max, MixedShape* plan,
               size_t* ws_bytes);
// Whether the tensor-core mixed decode serves these handles and T_max: d = 128,
// outlier parts of 32 channels, mse parts, instantiated bit pairs, T_max % 4 == 0.
// Zeroes n merge tickets in a kernel launched as a programmatic dependent,
// which lets the decode launched right after it (as its programmatic dependent)
// start while the kernels before finish; the decode's griddepcontrol.wait then
// covers every kernel before the clearing one (tq_decode.cu).
int launch_clear_tickets(int* tickets, int n, cudaStream_t s);
bool mixed_decode_tc_supported(const tq_ctx& hko, const tq_ctx& hkn, const tq_ctx& hvo, const tq_ctx& hvn,
                               int T_max);
int launch_mixed_decode(const MixedDecode& m, const MixedShape& p, cudaStream_t s);
int launch_select_outlier_channels(const void* x, int x_dtype, int64_t n_rows, int64_t stride, int d, int d_o,
                                   double* energy, int32_t* perm, cudaStream_t s);

// Decode-step append (tq_append.cu): quantize the new K and V rows [B·Hkv, d] into
// the next free token of each (batch, KV head) slab; the launch's last block then
// bumps the lengths and zeroes the decode's n_tickets merge tickets (if any).
// Behind the decode-step append, decode CTAs of at least this many tokens stream
// their rows below the pre-append length before waiting for the append, and the
// append runs on the SMs the decode grid leaves free when they suffice.  With
// shorter chunks the append would still be running when the CTAs finish that
// prefix, and the streaming only slows it down.
constexpr int kAppendStreamChunk = 4096;
// decode_ctas, decode_chunk: CTAs and tokens per CTA of the decode launched after
// the append (decode_split_ctas, the plan's chunk), which choose the append's grid.
int launch_append(const tq_ctx& hk, const tq_ctx& hv, const void* k_new, const void* v_new, int x_dtype, int B,
                  int Hkv, int T_max, int32_t* lens, const tq_planes& kc, const tq_planes& vc, int* tickets,
                  int n_tickets, int64_t decode_ctas, int decode_chunk, cudaStream_t s);
int launch_quantize_tc(const tq_ctx& h, const void* x, int x_dtype, int64_t n_rows, int64_t x_row_stride,
                       const tq_planes& out, cudaStream_t s);
// Two mse quantizers (same d ∈ {64, 128}, b, rotation kind) in one tensor-core launch.
bool quantize_pair_tc_supported(const tq_ctx& ha, const tq_ctx& hb, int x_dtype, int64_t rows_a, int64_t rows_b);
int launch_quantize_pair_tc(const tq_ctx& ha, const void* xa, int64_t rows_a, int64_t stride_a, const tq_planes& out_a,
                            const tq_ctx& hb, const void* xb, int64_t rows_b, int64_t stride_b, const tq_planes& out_b,
                            int x_dtype, cudaStream_t s);
int launch_quantize(const tq_ctx& h, const void* x, int x_dtype, int64_t n_rows,
                    int64_t x_row_stride, const tq_planes& out, cudaStream_t s);
int launch_dequantize(const tq_ctx& h, const tq_planes& in, int64_t n_rows, void* y,
                      int y_dtype, cudaStream_t s);

struct DecodeShape {
    int B, Hq, Hkv, T_max, d, G, n_splits, chunk;
};
int decode_plan(const tq_ctx& hk, const tq_ctx& hv, int B, int Hq, int Hkv, int T_max,
                DecodeShape* plan, size_t* ws_bytes);
// tickets_zeroed: the merge tickets (decode_tickets) were zeroed by the launch
// before this one, so the tensor-core path skips its own clearing.
int launch_decode(const tq_ctx& hk, const tq_ctx& hv, const DecodeShape& plan, const void* q,
                  int q_dtype, const tq_planes& kc, const tq_planes& vc,
                  const int32_t* seq_lens, float scale, float* out, float* scores_out,
                  void* workspace, cudaStream_t s, bool tickets_zeroed = false);
// The merge tickets of a decode workspace: where they lie and how many there are.
int* decode_tickets(const tq_ctx& hv, const DecodeShape& plan, void* workspace, int* count);
// CTAs of the split kernel of this plan.
int64_t decode_split_ctas(const DecodeShape& plan);

}  // namespace tq
