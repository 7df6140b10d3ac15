// C ABI entry points of libtq: argument validation, parameter upload, dispatch
// to the kernel launchers.  Declarations and contracts are in include/tq.h.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <new>

#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "tq_internal.h"

namespace tq {

static thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(TQ_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

namespace {

// Device allocations this thread has already validated: [base, end) on a device.
// A pointer inside one of them needs no attribute query (the query costs about
// a microsecond, and a call validates up to a dozen pointers).  Ranges come from
// the driver's allocation lookup; only plain device memory is remembered.
struct DevRange {
    uintptr_t base = 0, end = 0;
    int dev = -1;
};
constexpr int kRangeCache = 16;
thread_local DevRange g_ranges[kRangeCache];
thread_local int g_range_next = 0;

bool allocation_range(const void* p, uintptr_t* base, uintptr_t* end) {
    static PFN_cuMemGetAddressRange_v3020 get_range = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 3020, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_range = reinterpret_cast<PFN_cuMemGetAddressRange_v3020>(fn);
        cudaGetLastError();
    });
    if (get_range == nullptr) return false;
    CUdeviceptr b = 0;
    size_t n = 0;
    if (get_range(&b, &n, (CUdeviceptr)(uintptr_t)p) != CUDA_SUCCESS || n == 0) return false;
    *base = (uintptr_t)b;
    *end = (uintptr_t)b + n;
    return true;
}

}  // namespace

int check_device_ptr(const void* p, const char* name, bool required) {
    if (p == nullptr) {
        if (required) return fail(TQ_EINVAL, "%s is NULL", name);
        return TQ_OK;
    }
    if (((uintptr_t)p & 15u) != 0) return fail(TQ_EALIGN, "%s is not 16-byte aligned", name);
    int dev = -1;
    cudaGetDevice(&dev);
    const uintptr_t a = (uintptr_t)p;
    for (const DevRange& r : g_ranges)
        if (r.dev == dev && a >= r.base && a < r.end) return TQ_OK;
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(TQ_EINVAL, "%s is not a CUDA pointer (%s)", name, cudaGetErrorName(e));
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return fail(TQ_EINVAL, "%s is not device memory", name);
    if (attr.device != dev) return fail(TQ_EINVAL, "%s lives on device %d, current is %d", name, attr.device, dev);
    uintptr_t b = 0, end = 0;
    if (attr.type == cudaMemoryTypeDevice && allocation_range(p, &b, &end)) {
        g_ranges[g_range_next] = DevRange{b, end, dev};
        g_range_next = (g_range_next + 1) % kRangeCache;
    }
    return TQ_OK;
}

namespace {

// Scale σ ∈ [1, 2) for the f16 centroid tables of the tensor-core decode: the
// tables hold f16(σ·c_k) and the kernels divide σ back out in f32.  Choosing σ
// so that every σ·c_k lands close to an f16 value removes most of the rounding
// of the centroids (2^-12 relative at σ = 1), which the softmax would amplify.
float centroid_table_scale(const Codebook& cb) {
    float best_s = 1.f;
    double best_err = 1e30;
    for (int i = 0; i < (1 << 16); ++i) {
        const float sc = 1.f + (float)i / 65536.f;
        double err = 0.0;
        for (int k = 0; k < cb.levels; ++k) {
            const float v = sc * cb.c[k];
            if (v == 0.f) continue;
            const float r = __half2float(__float2half_rn(v));
            const double e = fabs((double)r - (double)v) / fabs((double)v);
            if (e > err) err = e;
        }
        if (err < best_err) {
            best_err = err;
            best_s = sc;
        }
    }
    return best_s;
}

// float → bfloat16 bits, round to nearest even (finite inputs).
uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

int upload(const std::vector<float>& host, float** dev) {
    cudaError_t e = cudaMalloc((void**)dev, host.size() * sizeof(float));
    if (e != cudaSuccess) {
        *dev = nullptr;
        cudaGetLastError();
        return fail(TQ_ENOMEM, "cudaMalloc of %zu bytes failed", host.size() * sizeof(float));
    }
    e = cudaMemcpy(*dev, host.data(), host.size() * sizeof(float), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy (parameter upload)");
    return TQ_OK;
}

void free_device(tq_ctx* h) {
    float** ptrs[] = {&h->dp.Pi, &h->dp.PiT, &h->dp.S, &h->dp.ST, &h->dp.TT};
    for (float** p : ptrs) {
        if (*p) cudaFree(*p);
        *p = nullptr;
    }
    uint16_t** hl[] = {&h->dp.Pi_hi,  &h->dp.Pi_lo,  &h->dp.S_hi,  &h->dp.S_lo, &h->dp.PiT_hi, &h->dp.PiT_lo,
                       &h->dp.ST_hi,  &h->dp.ST_lo,  &h->dp.T_hi,  &h->dp.T_lo, &h->dp.Pm};
    for (uint16_t** p : hl) {
        if (*p) cudaFree(*p);
        *p = nullptr;
    }
    if (h->dp.status) cudaFree(h->dp.status);
    h->dp.status = nullptr;
}

int upload_u16(const std::vector<uint16_t>& host, uint16_t** dev) {
    cudaError_t e = cudaMalloc((void**)dev, host.size() * sizeof(uint16_t));
    if (e != cudaSuccess) {
        *dev = nullptr;
        cudaGetLastError();
        return fail(TQ_ENOMEM, "cudaMalloc of %zu bytes failed", host.size() * sizeof(uint16_t));
    }
    e = cudaMemcpy(*dev, host.data(), host.size() * sizeof(uint16_t), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy (parameter upload)");
    return TQ_OK;
}

float bf16_bits_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

// M = M_hi + M_lo as two bf16 matrices (same row-major layout as M).
int upload_bf16_split(const std::vector<double>& m, uint16_t** dhi, uint16_t** dlo) {
    std::vector<uint16_t> hi(m.size()), lo(m.size());
    for (size_t k = 0; k < m.size(); ++k) {
        hi[k] = f32_to_bf16((float)m[k]);
        lo[k] = f32_to_bf16((float)(m[k] - (double)bf16_bits_to_f32(hi[k])));
    }
    int rc = upload_u16(hi, dhi);
    if (rc == TQ_OK) rc = upload_u16(lo, dlo);
    return rc;
}

std::vector<double> transposed(const std::vector<double>& m, int d) {
    std::vector<double> t(m.size());
    for (int j = 0; j < d; ++j)
        for (int i = 0; i < d; ++i) t[(size_t)i * d + j] = m[(size_t)j * d + i];
    return t;
}

// Π = Π_hi + Π_lo (and S = S_hi + S_lo) in bf16 for the tensor-core kernels, their
// transposes split the same way, plus the TMA maps over Π_hi / Π_lo.
int upload_tensor_core_params(tq_ctx* h) {
    const int d = h->hp.d;
    int rc = upload_bf16_split(h->hp.Pi, &h->dp.Pi_hi, &h->dp.Pi_lo);
    if (rc == TQ_OK && h->hp.variant == TQ_PROD) rc = upload_bf16_split(h->hp.S, &h->dp.S_hi, &h->dp.S_lo);
    if (rc == TQ_OK) rc = upload_bf16_split(transposed(h->hp.Pi, d), &h->dp.PiT_hi, &h->dp.PiT_lo);
    if (rc == TQ_OK && h->hp.variant == TQ_PROD)
        rc = upload_bf16_split(transposed(h->hp.S, d), &h->dp.ST_hi, &h->dp.ST_lo);
    if (rc != TQ_OK) return rc;
    if (d % 64 == 0) {
        rc = encode_tmap_bf16_2d(&h->dp.tm_pi_hi, h->dp.Pi_hi, d, d, (uint64_t)d * 2, 64, d);
        if (rc == TQ_OK) rc = encode_tmap_bf16_2d(&h->dp.tm_pi_lo, h->dp.Pi_lo, d, d, (uint64_t)d * 2, 64, d);
    }
    if (rc == TQ_OK && h->hp.rotation == TQ_ROT_HADAMARD) {
        // √d·Π has entries ±1: one exact bf16 operand, one MMA pass
        std::vector<uint16_t> pm((size_t)d * d);
        const double sd = sqrt((double)d);
        for (size_t k = 0; k < pm.size(); ++k) pm[k] = h->hp.Pi[k] * sd > 0.0 ? 0x3F80u : 0xBF80u;
        rc = upload_u16(pm, &h->dp.Pm);
        if (rc == TQ_OK && d % 64 == 0) rc = encode_tmap_bf16_2d(&h->dp.tm_pm, h->dp.Pm, d, d, (uint64_t)d * 2, 64, d);
        h->rot_passes = 1;
        h->rot_norm_scale = (float)(1.0 / sd);
    }
    if (rc == TQ_OK && h->hp.variant == TQ_PROD) {
        // T = S·Πᵀ (T_ij = Σ_k S_ik Π_jk) as f16 hi + lo, row-major [i][j]: the operand of
        // the QJL sketch s = T·e of the rotated residual e
        std::vector<uint16_t> thi((size_t)d * d), tlo((size_t)d * d);
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) {
                double acc = 0.0;
                for (int k = 0; k < d; ++k) acc += h->hp.S[(size_t)i * d + k] * h->hp.Pi[(size_t)j * d + k];
                const __half vh = __float2half_rn((float)acc);
                const __half vl = __float2half_rn((float)(acc - (double)__half2float(vh)));
                thi[(size_t)i * d + j] = __half_as_ushort(vh);
                tlo[(size_t)i * d + j] = __half_as_ushort(vl);
            }
        rc = upload_u16(thi, &h->dp.T_hi);
        if (rc == TQ_OK) rc = upload_u16(tlo, &h->dp.T_lo);
        if (rc == TQ_OK && d % 64 == 0) {
            rc = encode_tmap_f16_2d(&h->dp.tm_t_hi, h->dp.T_hi, d, d, (uint64_t)d * 2, 64, d);
            if (rc == TQ_OK) rc = encode_tmap_f16_2d(&h->dp.tm_t_lo, h->dp.T_lo, d, d, (uint64_t)d * 2, 64, d);
        }
    }
    return rc;
}

int upload_params(tq_ctx* h) {
    const HostParams& hp = h->hp;
    const int d = hp.d;
    std::vector<float> a((size_t)d * d), b((size_t)d * d);
    for (int j = 0; j < d; ++j)
        for (int i = 0; i < d; ++i) {
            a[(size_t)j * d + i] = (float)hp.Pi[(size_t)j * d + i];
            b[(size_t)i * d + j] = (float)hp.Pi[(size_t)j * d + i];
        }
    int rc = upload(a, &h->dp.Pi);
    if (rc == TQ_OK) rc = upload(b, &h->dp.PiT);
    if (rc == TQ_OK && hp.variant == TQ_PROD) {
        for (int j = 0; j < d; ++j)
            for (int i = 0; i < d; ++i) {
                a[(size_t)j * d + i] = (float)hp.S[(size_t)j * d + i];
                b[(size_t)i * d + j] = (float)hp.S[(size_t)j * d + i];
            }
        rc = upload(a, &h->dp.S);
        if (rc == TQ_OK) rc = upload(b, &h->dp.ST);
        if (rc == TQ_OK) {
            // T = S Πᵀ, stored transposed: TT[j*d+i] = T_ij = Σ_k S_ik Π_jk
            for (int i = 0; i < d; ++i)
                for (int j = 0; j < d; ++j) {
                    double acc = 0.0;
                    for (int k = 0; k < d; ++k) acc += hp.S[(size_t)i * d + k] * hp.Pi[(size_t)j * d + k];
                    a[(size_t)j * d + i] = (float)acc;
                }
            rc = upload(a, &h->dp.TT);
        }
    }
    if (rc == TQ_OK) rc = upload_tensor_core_params(h);
    if (rc == TQ_OK) {
        cudaError_t e = cudaMalloc((void**)&h->dp.status, 2 * sizeof(int));
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(TQ_ENOMEM, "cudaMalloc of the status word failed");
        }
        e = cudaMemset(h->dp.status, 0, 2 * sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset (status word)");
        h->dp.append_done = h->dp.status + 1;
    }
    return rc;
}

int validate_handle(tq_handle h, const char* name) {
    if (h == nullptr) return fail(TQ_EINVAL, "%s handle is NULL", name);
    int dev = -1;
    cudaGetDevice(&dev);
    if (dev != h->device) return fail(TQ_EINVAL, "%s handle was created on device %d, current is %d", name, h->device, dev);
    return TQ_OK;
}

int check_planes(const tq_ctx& h, const tq_planes& p, const char* what) {
    char nm[64];
    int rc;
    if (h.code_bytes > 0) {
        snprintf(nm, sizeof nm, "%s.codes", what);
        if ((rc = check_device_ptr(p.codes, nm, true)) != TQ_OK) return rc;
    }
    snprintf(nm, sizeof nm, "%s.norm", what);
    if ((rc = check_device_ptr(p.norm, nm, true)) != TQ_OK) return rc;
    if (h.hp.variant == TQ_PROD) {
        snprintf(nm, sizeof nm, "%s.signs", what);
        if ((rc = check_device_ptr(p.signs, nm, true)) != TQ_OK) return rc;
        snprintf(nm, sizeof nm, "%s.rnorm", what);
        if ((rc = check_device_ptr(p.rnorm, nm, true)) != TQ_OK) return rc;
    }
    return TQ_OK;
}

}  // namespace

namespace {
int encode_tmap_2d(CUtensorMapDataType dtype, CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (encode == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
            cudaGetLastError();
            return fail(TQ_ECUDA, "cuTensorMapEncodeTiled entry point unavailable");
        }
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(TQ_ECUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return TQ_OK;
}
}  // namespace

int encode_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    return encode_tmap_2d(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, map, base, inner, outer, row_stride_bytes, box_inner,
                          box_outer);
}
int encode_tmap_f16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                       uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    return encode_tmap_2d(CU_TENSOR_MAP_DATA_TYPE_FLOAT16, map, base, inner, outer, row_stride_bytes, box_inner,
                          box_outer);
}

}  // namespace tq

using namespace tq;

extern "C" {

const char* tq_last_error(void) { return g_err; }

int tq_build_params_host(int d, int bits, int variant, uint64_t seed, double* Pi, double* S,
                         double* centroids, double* bounds) {
    return tq_build_params_host_ex(d, bits, variant, TQ_ROT_QR, seed, Pi, S, centroids, bounds);
}

int tq_build_params_host_ex(int d, int bits, int variant, int rotation, uint64_t seed, double* Pi, double* S,
                            double* centroids, double* bounds) {
    HostParams hp;
    int rc = build_host_params(d, bits, variant, rotation, seed, &hp);
    if (rc != TQ_OK) return rc;
    if (Pi) memcpy(Pi, hp.Pi.data(), hp.Pi.size() * sizeof(double));
    if (S && variant == TQ_PROD) memcpy(S, hp.S.data(), hp.S.size() * sizeof(double));
    if (centroids) memcpy(centroids, hp.centroids.data(), hp.centroids.size() * sizeof(double));
    if (bounds && !hp.bounds.empty()) memcpy(bounds, hp.bounds.data(), hp.bounds.size() * sizeof(double));
    g_err[0] = 0;
    return TQ_OK;
}

int tq_init(int d, int bits, int variant, uint64_t seed, tq_handle* out) {
    return tq_init_ex(d, bits, variant, TQ_ROT_QR, seed, out);
}

int tq_init_ex(int d, int bits, int variant, int rotation, uint64_t seed, tq_handle* out) {
    if (out == nullptr) return fail(TQ_EINVAL, "out is NULL");
    *out = nullptr;
    tq_ctx* h = new (std::nothrow) tq_ctx();
    if (!h) return fail(TQ_ENOMEM, "host allocation failed");
    int rc = build_host_params(d, bits, variant, rotation, seed, &h->hp);
    if (rc != TQ_OK) {
        delete h;
        return rc;
    }
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) {
        delete h;
        return cuda_fail(e, "cudaGetDevice");
    }
    if ((e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device)) != cudaSuccess) {
        delete h;
        return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    }
    h->code_bytes = h->hp.b_mse * d / 8;
    h->sign_bytes = variant == TQ_PROD ? d / 8 : 0;
    h->gamma = (float)(sqrt(M_PI / 2.0) / d);
    memset(&h->cb, 0, sizeof(h->cb));
    h->cb.levels = h->hp.levels;
    for (int i = 0; i < h->hp.levels; ++i) h->cb.c[i] = (float)h->hp.centroids[i];
    for (int i = 0; i + 1 < h->hp.levels; ++i) h->cb.t[i] = (float)h->hp.bounds[i];
    h->cb.lut_scale = centroid_table_scale(h->cb);
    rc = upload_params(h);
    if (rc != TQ_OK) {
        free_device(h);
        delete h;
        return rc;
    }
    *out = h;
    g_err[0] = 0;
    return TQ_OK;
}

int tq_destroy(tq_handle h) {
    if (h == nullptr) return TQ_OK;
    free_device(h);
    delete h;
    return TQ_OK;
}

int tq_row_bytes(tq_handle h, int* code_bytes, int* sign_bytes) {
    if (h == nullptr) return fail(TQ_EINVAL, "handle is NULL");
    if (code_bytes) *code_bytes = h->code_bytes;
    if (sign_bytes) *sign_bytes = h->sign_bytes;
    return TQ_OK;
}

int tq_device_status(tq_handle h, int* status, int clear) {
    int rc = validate_handle(h, "quantizer");
    if (rc != TQ_OK) return rc;
    if (status == nullptr) return fail(TQ_EINVAL, "status is NULL");
    cudaError_t e = cudaMemcpy(status, h->dp.status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
    if (clear && *status != 0) {
        e = cudaMemset(h->dp.status, 0, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    }
    return TQ_OK;
}

int tq_check_wait_timeout(tq_handle h, int code, uint64_t limit_ns, void* stream) {
    int rc = validate_handle(h, "quantizer");
    if (rc != TQ_OK) return rc;
    if (code < 1 || code > 1000) return fail(TQ_EINVAL, "code must be in [1, 1000]");
    if (limit_ns < 1 || limit_ns > 1000000000ull) return fail(TQ_EINVAL, "limit_ns must be in [1, 1e9]");
    return launch_expire_wait(*h, code, limit_ns, (cudaStream_t)stream);
}

int tq_get_params(tq_handle h, double* Pi, double* S, double* centroids, double* bounds) {
    if (h == nullptr) return fail(TQ_EINVAL, "handle is NULL");
    const HostParams& hp = h->hp;
    if (Pi) memcpy(Pi, hp.Pi.data(), hp.Pi.size() * sizeof(double));
    if (S && hp.variant == TQ_PROD) memcpy(S, hp.S.data(), hp.S.size() * sizeof(double));
    if (centroids) memcpy(centroids, hp.centroids.data(), hp.centroids.size() * sizeof(double));
    if (bounds && !hp.bounds.empty()) memcpy(bounds, hp.bounds.data(), hp.bounds.size() * sizeof(double));
    return TQ_OK;
}

namespace {

int check_quantize_args(tq_handle h, const void* x, int x_dtype, int64_t n_rows, int64_t x_row_stride,
                        const tq_planes& out, const char* what) {
    int rc = validate_handle(h, what);
    if (rc != TQ_OK) return rc;
    if (n_rows < 0) return fail(TQ_EINVAL, "n_rows=%lld is negative", (long long)n_rows);
    if (x_dtype != TQ_BF16 && x_dtype != TQ_F32) return fail(TQ_EINVAL, "x_dtype=%d invalid", x_dtype);
    if (n_rows == 0) return TQ_OK;
    const int d = h->hp.d;
    const int es = x_dtype == TQ_BF16 ? 2 : 4;
    if (x_row_stride < d) return fail(TQ_EINVAL, "x_row_stride=%lld < d=%d", (long long)x_row_stride, d);
    if ((x_row_stride * es) % 16 != 0) return fail(TQ_EALIGN, "x_row_stride*elem_size must be a multiple of 16 bytes");
    if ((rc = check_device_ptr(x, "x", true)) != TQ_OK) return rc;
    return check_planes(*h, out, "out");
}

}  // namespace

int tq_quantize(tq_handle h, const void* x, int x_dtype, int64_t n_rows, int64_t x_row_stride,
                tq_planes out, void* stream) {
    const int rc = check_quantize_args(h, x, x_dtype, n_rows, x_row_stride, out, "quantizer");
    if (rc != TQ_OK || n_rows == 0) return rc;
    return launch_quantize(*h, x, x_dtype, n_rows, x_row_stride, out, (cudaStream_t)stream);
}

int tq_quantize_kv(tq_handle hk, tq_handle hv, const void* k, const void* v, int x_dtype, int64_t k_rows,
                   int64_t v_rows, int64_t k_row_stride, int64_t v_row_stride, tq_planes k_out, tq_planes v_out,
                   void* stream) {
    int rc = check_quantize_args(hk, k, x_dtype, k_rows, k_row_stride, k_out, "key quantizer");
    if (rc != TQ_OK) return rc;
    if ((rc = check_quantize_args(hv, v, x_dtype, v_rows, v_row_stride, v_out, "value quantizer")) != TQ_OK) return rc;
    const cudaStream_t s = (cudaStream_t)stream;
    if (quantize_pair_tc_supported(*hk, *hv, x_dtype, k_rows, v_rows))
        return launch_quantize_pair_tc(*hk, k, k_rows, k_row_stride, k_out, *hv, v, v_rows, v_row_stride, v_out,
                                       x_dtype, s);
    if (k_rows > 0 && (rc = launch_quantize(*hk, k, x_dtype, k_rows, k_row_stride, k_out, s)) != TQ_OK) return rc;
    if (v_rows > 0) rc = launch_quantize(*hv, v, x_dtype, v_rows, v_row_stride, v_out, s);
    return rc;
}

int tq_dequantize(tq_handle h, tq_planes in, int64_t n_rows, void* y, int y_dtype, void* stream) {
    int rc = validate_handle(h, "quantizer");
    if (rc != TQ_OK) return rc;
    if (n_rows < 0) return fail(TQ_EINVAL, "n_rows=%lld is negative", (long long)n_rows);
    if (y_dtype != TQ_BF16 && y_dtype != TQ_F32) return fail(TQ_EINVAL, "y_dtype=%d invalid", y_dtype);
    if (n_rows == 0) return TQ_OK;
    if ((rc = check_device_ptr(y, "y", true)) != TQ_OK) return rc;
    if ((rc = check_planes(*h, in, "in")) != TQ_OK) return rc;
    return launch_dequantize(*h, in, n_rows, y, y_dtype, (cudaStream_t)stream);
}

int tq_decode_workspace_bytes(tq_handle hk, tq_handle hv, int B, int Hq, int Hkv, int T_max, size_t* bytes) {
    if (bytes == nullptr) return fail(TQ_EINVAL, "bytes is NULL");
    int rc = validate_handle(hk, "key");
    if (rc == TQ_OK) rc = validate_handle(hv, "value");
    if (rc != TQ_OK) return rc;
    DecodeShape plan;
    return decode_plan(*hk, *hv, B, Hq, Hkv, T_max, &plan, bytes);
}

int tq_decode_attention(tq_handle hk, tq_handle hv, const void* q, int q_dtype, tq_planes kc,
                        tq_planes vc, const int32_t* seq_lens, int B, int Hq, int Hkv, int T_max,
                        float scale, float* out, float* scores_out, void* workspace, size_t ws_bytes,
                        void* stream) {
    int rc = validate_handle(hk, "key");
    if (rc == TQ_OK) rc = validate_handle(hv, "value");
    if (rc != TQ_OK) return rc;
    if (q_dtype != TQ_BF16 && q_dtype != TQ_F32) return fail(TQ_EINVAL, "q_dtype=%d invalid", q_dtype);
    DecodeShape plan;
    size_t need = 0;
    if ((rc = decode_plan(*hk, *hv, B, Hq, Hkv, T_max, &plan, &need)) != TQ_OK) return rc;
    if (B == 0 || Hq == 0) return TQ_OK;
    if (ws_bytes < need) return fail(TQ_EWORKSPACE, "workspace of %zu bytes < required %zu", ws_bytes, need);
    if ((rc = check_device_ptr(q, "q", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(seq_lens, "seq_lens", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(out, "out", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(scores_out, "scores_out", false)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(workspace, "workspace", true)) != TQ_OK) return rc;
    if (T_max > 0) {
        if ((rc = check_planes(*hk, kc, "kc")) != TQ_OK) return rc;
        if ((rc = check_planes(*hv, vc, "vc")) != TQ_OK) return rc;
    }
    if (scale <= 0.f) scale = (float)(1.0 / sqrt((double)hk->hp.d));
    return launch_decode(*hk, *hv, plan, q, q_dtype, kc, vc, seq_lens, scale, out, scores_out, workspace,
                         (cudaStream_t)stream);
}

int tq_select_outlier_channels(const void* x, int x_dtype, int64_t n_rows, int64_t x_row_stride, int d, int d_o,
                               double* energy, int32_t* perm, void* stream) {
    if (x_dtype != TQ_BF16 && x_dtype != TQ_F32) return fail(TQ_EINVAL, "x_dtype=%d invalid", x_dtype);
    if (d < 2 * kMinD || d > kMaxD || d % 32 != 0) return fail(TQ_EUNSUPPORTED, "d=%d unsupported (64..256, multiple of 32)", d);
    if (d_o < kMinD || d_o > d - kMinD || d_o % 32 != 0)
        return fail(TQ_EINVAL, "d_o=%d must be a multiple of 32 in [32, d − 32]", d_o);
    if (n_rows < 0) return fail(TQ_EINVAL, "n_rows=%lld is negative", (long long)n_rows);
    const int es = x_dtype == TQ_BF16 ? 2 : 4;
    if (x_row_stride < d) return fail(TQ_EINVAL, "x_row_stride=%lld < d=%d", (long long)x_row_stride, d);
    if ((x_row_stride * es) % 16 != 0) return fail(TQ_EALIGN, "x_row_stride*elem_size must be a multiple of 16 bytes");
    int rc;
    if (n_rows > 0 && (rc = check_device_ptr(x, "x", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(energy, "energy", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(perm, "perm", true)) != TQ_OK) return rc;
    return launch_select_outlier_channels(x, x_dtype, n_rows, x_row_stride, d, d_o, energy, perm,
                                          (cudaStream_t)stream);
}

namespace {
int validate_split(tq_handle ho, tq_handle hn, const char* what) {
    int rc = validate_handle(ho, what);
    if (rc == TQ_OK) rc = validate_handle(hn, what);
    if (rc != TQ_OK) return rc;
    if (ho->hp.variant != hn->hp.variant) return fail(TQ_EINVAL, "%s parts differ in variant", what);
    if (ho->hp.d + hn->hp.d > kMaxD) return fail(TQ_EUNSUPPORTED, "%s parts sum to d=%d > %d", what,
                                                 ho->hp.d + hn->hp.d, kMaxD);
    return TQ_OK;
}
}  // namespace

size_t tq_mixed_quantize_scratch_bytes(void) { return mixed_tc_scratch_bytes(); }

namespace {
// The argument checks of one mixed quantize side (rows, perm, planes); n_rows = 0
// checks only the handles and the dtype.
int check_mixed_quantize_args(tq_handle ho, tq_handle hn, const int32_t* perm, const void* x, int x_dtype,
                              int64_t n_rows, int64_t x_row_stride, const tq_planes& out_o, const tq_planes& out_n,
                              const char* what) {
    int rc = validate_split(ho, hn, what);
    if (rc != TQ_OK) return rc;
    if (n_rows < 0) return fail(TQ_EINVAL, "%s: n_rows=%lld is negative", what, (long long)n_rows);
    if (x_dtype != TQ_BF16 && x_dtype != TQ_F32) return fail(TQ_EINVAL, "x_dtype=%d invalid", x_dtype);
    if (n_rows == 0) return TQ_OK;
    const int d = ho->hp.d + hn->hp.d;
    const int es = x_dtype == TQ_BF16 ? 2 : 4;
    if (x_row_stride < d)
        return fail(TQ_EINVAL, "%s: x_row_stride=%lld < d=%d", what, (long long)x_row_stride, d);
    if ((x_row_stride * es) % 16 != 0)
        return fail(TQ_EALIGN, "%s: x_row_stride*elem_size must be a multiple of 16 bytes", what);
    if ((rc = check_device_ptr(perm, "perm", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(x, "x", true)) != TQ_OK) return rc;
    if ((rc = check_planes(*ho, out_o, "out_o")) != TQ_OK) return rc;
    return check_planes(*hn, out_n, "out_n");
}

// One side after its checks (n_rows > 0).
int mixed_quantize_side(tq_handle ho, tq_handle hn, const int32_t* perm, const void* x, int x_dtype, int64_t n_rows,
                        int64_t x_row_stride, const tq_planes& out_o, const tq_planes& out_n, void* scratch,
                        size_t scratch_bytes, cudaStream_t s) {
    if (mixed_quantize_tc_supported(*ho, *hn, x_dtype, n_rows, x_row_stride, scratch, scratch_bytes))
        return launch_mixed_quantize_tc(*ho, *hn, perm, x, n_rows, x_row_stride, out_o, out_n, scratch, s);
    const int d = ho->hp.d + hn->hp.d;
    int rc = launch_quantize_part(*ho, x, x_dtype, n_rows, x_row_stride, perm, d, out_o, s);
    if (rc == TQ_OK) rc = launch_quantize_part(*hn, x, x_dtype, n_rows, x_row_stride, perm + ho->hp.d, d, out_n, s);
    return rc;
}
}  // namespace

int tq_mixed_quantize(tq_handle ho, tq_handle hn, const int32_t* perm, const void* x, int x_dtype, int64_t n_rows,
                      int64_t x_row_stride, tq_planes out_o, tq_planes out_n, void* scratch, size_t scratch_bytes,
                      void* stream) {
    int rc = check_mixed_quantize_args(ho, hn, perm, x, x_dtype, n_rows, x_row_stride, out_o, out_n, "quantizer");
    if (rc != TQ_OK || n_rows == 0) return rc;
    if ((rc = check_device_ptr(scratch, "scratch", false)) != TQ_OK) return rc;
    return mixed_quantize_side(ho, hn, perm, x, x_dtype, n_rows, x_row_stride, out_o, out_n, scratch, scratch_bytes,
                               (cudaStream_t)stream);
}

int tq_mixed_quantize_kv(tq_handle hko, tq_handle hkn, tq_handle hvo, tq_handle hvn, const int32_t* perm_k,
                         const int32_t* perm_v, const void* k, const void* v, int x_dtype, int64_t k_rows,
                         int64_t v_rows, int64_t k_row_stride, int64_t v_row_stride, tq_planes k_out_o,
                         tq_planes k_out_n, tq_planes v_out_o, tq_planes v_out_n, void* scratch,
                         size_t scratch_bytes, void* stream) {
    int rc = check_mixed_quantize_args(hko, hkn, perm_k, k, x_dtype, k_rows, k_row_stride, k_out_o, k_out_n, "key");
    if (rc != TQ_OK) return rc;
    rc = check_mixed_quantize_args(hvo, hvn, perm_v, v, x_dtype, v_rows, v_row_stride, v_out_o, v_out_n, "value");
    if (rc != TQ_OK) return rc;
    if ((rc = check_device_ptr(scratch, "scratch", false)) != TQ_OK) return rc;
    const cudaStream_t s = (cudaStream_t)stream;
    if (k_rows > 0 && v_rows > 0 &&
        mixed_quantize_pair_tc_supported(*hko, *hkn, *hvo, *hvn, x_dtype, k_rows, k_row_stride, v_rows, v_row_stride,
                                         scratch, scratch_bytes))
        return launch_mixed_quantize_pair_tc(*hko, *hkn, *hvo, *hvn, perm_k, perm_v, k, v, k_rows, k_row_stride,
                                             v_rows, v_row_stride, k_out_o, k_out_n, v_out_o, v_out_n, scratch, s);
    // two calls in stream order, so they may share the scratch
    if (k_rows > 0 && (rc = mixed_quantize_side(hko, hkn, perm_k, k, x_dtype, k_rows, k_row_stride, k_out_o, k_out_n,
                                                scratch, scratch_bytes, s)) != TQ_OK)
        return rc;
    if (v_rows > 0)
        rc = mixed_quantize_side(hvo, hvn, perm_v, v, x_dtype, v_rows, v_row_stride, v_out_o, v_out_n, scratch,
                                 scratch_bytes, s);
    return rc;
}

int tq_mixed_dequantize(tq_handle ho, tq_handle hn, const int32_t* perm, tq_planes in_o, tq_planes in_n,
                        int64_t n_rows, void* y, int y_dtype, void* stream) {
    int rc = validate_split(ho, hn, "quantizer");
    if (rc != TQ_OK) return rc;
    if (n_rows < 0) return fail(TQ_EINVAL, "n_rows=%lld is negative", (long long)n_rows);
    if (y_dtype != TQ_BF16 && y_dtype != TQ_F32) return fail(TQ_EINVAL, "y_dtype=%d invalid", y_dtype);
    if (n_rows == 0) return TQ_OK;
    const int d = ho->hp.d + hn->hp.d;
    if ((rc = check_device_ptr(perm, "perm", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(y, "y", true)) != TQ_OK) return rc;
    if ((rc = check_planes(*ho, in_o, "in_o")) != TQ_OK) return rc;
    if ((rc = check_planes(*hn, in_n, "in_n")) != TQ_OK) return rc;
    const cudaStream_t s = (cudaStream_t)stream;
    rc = launch_dequantize_part(*ho, in_o, n_rows, perm, d, y, y_dtype, s);
    if (rc == TQ_OK) rc = launch_dequantize_part(*hn, in_n, n_rows, perm + ho->hp.d, d, y, y_dtype, s);
    return rc;
}

namespace {
int mixed_shape(tq_handle hko, tq_handle hkn, tq_handle hvo, tq_handle hvn, int B, int Hq, int Hkv, int T_max,
                MixedShape* plan, size_t* bytes) {
    int rc = validate_split(hko, hkn, "key");
    if (rc == TQ_OK) rc = validate_split(hvo, hvn, "value");
    if (rc != TQ_OK) return rc;
    const int d = hko->hp.d + hkn->hp.d;
    if (hvo->hp.d + hvn->hp.d != d) return fail(TQ_EINVAL, "key d=%d and value d=%d differ", d,
                                                hvo->hp.d + hvn->hp.d);
    const bool tc = mixed_decode_tc_supported(*hko, *hkn, *hvo, *hvn, T_max);
    return mixed_plan(d, hko->num_sms, hvo->hp.variant == TQ_PROD, tc, B, Hq, Hkv, T_max, plan, bytes);
}
}  // namespace

int tq_mixed_decode_workspace_bytes(tq_handle hko, tq_handle hkn, tq_handle hvo, tq_handle hvn, int B, int Hq,
                                    int Hkv, int T_max, size_t* bytes) {
    if (bytes == nullptr) return fail(TQ_EINVAL, "bytes is NULL");
    MixedShape plan;
    return mixed_shape(hko, hkn, hvo, hvn, B, Hq, Hkv, T_max, &plan, bytes);
}

int tq_mixed_decode_attention(tq_handle hko, tq_handle hkn, tq_handle hvo, tq_handle hvn, const int32_t* perm_k,
                              const int32_t* perm_v, const void* q, int q_dtype, tq_planes kc_o, tq_planes kc_n,
                              tq_planes vc_o, tq_planes vc_n, const int32_t* seq_lens, int B, int Hq, int Hkv,
                              int T_max, float scale, float* out, float* scores_out, void* workspace,
                              size_t ws_bytes, void* stream) {
    if (q_dtype != TQ_BF16 && q_dtype != TQ_F32) return fail(TQ_EINVAL, "q_dtype=%d invalid", q_dtype);
    MixedShape plan;
    size_t need = 0;
    int rc = mixed_shape(hko, hkn, hvo, hvn, B, Hq, Hkv, T_max, &plan, &need);
    if (rc != TQ_OK) return rc;
    if (B == 0 || Hq == 0) return TQ_OK;
    if (ws_bytes < need) return fail(TQ_EWORKSPACE, "workspace of %zu bytes < required %zu", ws_bytes, need);
    if ((rc = check_device_ptr(perm_k, "perm_k", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(perm_v, "perm_v", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(q, "q", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(seq_lens, "seq_lens", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(out, "out", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(scores_out, "scores_out", false)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(workspace, "workspace", true)) != TQ_OK) return rc;
    if (T_max > 0) {
        if ((rc = check_planes(*hko, kc_o, "kc_o")) != TQ_OK) return rc;
        if ((rc = check_planes(*hkn, kc_n, "kc_n")) != TQ_OK) return rc;
        if ((rc = check_planes(*hvo, vc_o, "vc_o")) != TQ_OK) return rc;
        if ((rc = check_planes(*hvn, vc_n, "vc_n")) != TQ_OK) return rc;
    }
    if (scale <= 0.f) scale = (float)(1.0 / sqrt((double)plan.d));
    MixedDecode m;
    m.hk[0] = hko; m.hk[1] = hkn; m.hv[0] = hvo; m.hv[1] = hvn;
    m.perm_k = perm_k; m.perm_v = perm_v;
    m.q = q; m.q_dtype = q_dtype;
    m.kc[0] = kc_o; m.kc[1] = kc_n; m.vc[0] = vc_o; m.vc[1] = vc_n;
    m.seq_lens = seq_lens; m.scale = scale; m.out = out; m.scores = scores_out; m.workspace = workspace;
    return launch_mixed_decode(m, plan, (cudaStream_t)stream);
}

int tq_decode_append_attention(tq_handle hk, tq_handle hv, const void* q, int q_dtype, const void* k_new,
                               const void* v_new, int kv_dtype, tq_planes kc, tq_planes vc, int32_t* seq_lens,
                               int B, int Hq, int Hkv, int T_max, float scale, float* out, void* workspace,
                               size_t ws_bytes, void* stream) {
    int rc = validate_handle(hk, "key");
    if (rc == TQ_OK) rc = validate_handle(hv, "value");
    if (rc != TQ_OK) return rc;
    if (q_dtype != TQ_BF16 && q_dtype != TQ_F32) return fail(TQ_EINVAL, "q_dtype=%d invalid", q_dtype);
    if (kv_dtype != TQ_BF16 && kv_dtype != TQ_F32) return fail(TQ_EINVAL, "kv_dtype=%d invalid", kv_dtype);
    DecodeShape plan;
    size_t need = 0;
    if ((rc = decode_plan(*hk, *hv, B, Hq, Hkv, T_max, &plan, &need)) != TQ_OK) return rc;
    if (B == 0 || Hq == 0) return TQ_OK;
    if (T_max <= 0) return fail(TQ_EINVAL, "T_max=%d leaves no room to append", T_max);
    if (ws_bytes < need) return fail(TQ_EWORKSPACE, "workspace of %zu bytes < required %zu", ws_bytes, need);
    if ((rc = check_device_ptr(q, "q", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(k_new, "k_new", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(v_new, "v_new", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(seq_lens, "seq_lens", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(out, "out", true)) != TQ_OK) return rc;
    if ((rc = check_device_ptr(workspace, "workspace", true)) != TQ_OK) return rc;
    if ((rc = check_planes(*hk, kc, "kc")) != TQ_OK) return rc;
    if ((rc = check_planes(*hv, vc, "vc")) != TQ_OK) return rc;
    if (scale <= 0.f) scale = (float)(1.0 / sqrt((double)hk->hp.d));
    const cudaStream_t s = (cudaStream_t)stream;
    int n_tickets = 0;
    int* tickets = decode_tickets(*hv, plan, workspace, &n_tickets);
    if ((rc = launch_append(*hk, *hv, k_new, v_new, kv_dtype, B, Hkv, T_max, seq_lens, kc, vc, tickets, n_tickets,
                            decode_split_ctas(plan), plan.chunk, s)) != TQ_OK)
        return rc;
    return launch_decode(*hk, *hv, plan, q, q_dtype, kc, vc, seq_lens, scale, out, nullptr, workspace, s, true);
}

}  // extern "C"
