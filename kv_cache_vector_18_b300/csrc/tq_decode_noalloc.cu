// tq_decode_attention_noalloc: decode attention for callers that cannot
// allocate device memory.  The workspace tq_decode_attention asks its caller
// for lives instead in one file-scope __device__ array of fixed size that every
// call on a device shares.
#include <atomic>
#include <mutex>

#include "tq_internal.h"

namespace {

// The shared scratch buffer.  In host code `g_decode_scratch` only names a
// host-side stand-in: its device address must be looked up with
// cudaGetSymbolAddress, once per device, with that device current.
static __device__ __align__(256) unsigned char g_decode_scratch[TQ_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
std::atomic<void*> g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch buffer on the current device.  The first call
// made with a device current looks it up (under a mutex); later calls read the
// cached address without taking the lock.
int scratch_on_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return tq::cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return tq::fail(TQ_EUNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        std::lock_guard<std::mutex> lock(g_mu);
        p = g_scratch_addr[dev].load(std::memory_order_relaxed);
        if (p == nullptr) {
            e = cudaGetSymbolAddress(&p, g_decode_scratch);
            if (e != cudaSuccess) return tq::cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
            g_scratch_addr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return TQ_OK;
}

}  // namespace

extern "C" int tq_decode_attention_noalloc(tq_handle hk, tq_handle hv, const void* q, int q_dtype,
                                           tq_planes kc, tq_planes vc, const int32_t* seq_lens, int B,
                                           int Hq, int Hkv, int T_max, float scale, float* out,
                                           float* scores_out, void* stream) {
    size_t need = 0;
    int rc = tq_decode_workspace_bytes(hk, hv, B, Hq, Hkv, T_max, &need);
    if (rc != TQ_OK) return rc;
    if (need > (size_t)TQ_NOALLOC_WORKSPACE_BYTES)
        return tq::fail(TQ_EWORKSPACE,
                        "these shapes need %zu bytes of decode scratch, more than the %u-byte static buffer of "
                        "tq_decode_attention_noalloc; call tq_decode_attention with a caller-owned workspace",
                        need, (unsigned)TQ_NOALLOC_WORKSPACE_BYTES);
    void* ws = nullptr;
    if ((rc = scratch_on_current_device(&ws)) != TQ_OK) return rc;
    // Nothing in the scratch needs clearing: every launch writes all of the
    // workspace it later reads (rotated queries and every split's partials).
    return tq_decode_attention(hk, hv, q, q_dtype, kc, vc, seq_lens, B, Hq, Hkv, T_max, scale, out, scores_out,
                               ws, (size_t)TQ_NOALLOC_WORKSPACE_BYTES, stream);
}
