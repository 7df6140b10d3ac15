/*
 * tq.h — C ABI of the TurboQuant KV-cache codec and compressed-cache decode
 * attention for NVIDIA B300 (sm_103a).
 *
 * Method: "Вечная математика TurboQuant: как сжать KV-кэш до предела Шеннона"
 * (blog.sergeynikolenko.ru/?p=11266).  Section names below are that page's:
 *   «Шаг 0» norm split, «Шаг 1» random rotation Π, «Шаг 2» Lloyd–Max codebook
 *   and nearest-centroid indices, «QJL» 1-bit sketch sign(S·x) with dequantizer
 *   √(π/2)/d·Sᵀz, «Собственно TurboQuant» (prod: (b−1)-bit mse + QJL of the
 *   residual, storing sign(S·r) and ‖r‖), Theorem 2 (the prod map).
 * The decode-attention consumer is the "custom attention kernel" the
 * nahornyi.ai commentary says the prod variant needs.  Also from that page:
 * «Что сделало сообщество» finding #3 (a Walsh–Hadamard rotation for the MSE
 * stage with an independent QJL transform: tq_init_ex), and the experiments
 * section's outlier-channel split (32 channels at 3 bits, 96 at 2: tq_mixed_*).
 * The decode step with append (tq_decode_append_attention) is this library's
 * serving entry point; the pages define no such step.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Return value: TQ_OK (0) or a negative TQ_E* code; tq_last_error() gives a
 *   thread-local message for the last failure on the calling thread.  No C++
 *   exception crosses this boundary and no kernel traps: invalid arguments are
 *   rejected on the host before any launch.
 * - "device pointer" arguments must point to memory of the current CUDA device
 *   (cudaMalloc / torch allocations) and be 16-byte aligned, else TQ_EALIGN or
 *   TQ_EINVAL.  The caller owns every buffer passed in; the library allocates
 *   device memory only inside tq_init and frees it in tq_destroy.
 * - `stream` is a cudaStream_t (NULL = legacy default stream).  All compute calls
 *   are asynchronous on that stream; they return after enqueueing.
 * - A handle may be used from several threads for compute calls concurrently;
 *   tq_destroy must not race with any other call on that handle.
 *
 * Packed cache planes (layout owned by this library; the pages leave it open)
 * --------------------------------------------------------------------------
 * For a handle with head dimension d, bits b and variant v, let b_m = b (mse) or
 * b − 1 (prod).  A row of the cache is stored across up to four planes, each a
 * dense array of n_rows equal-sized records (record i at byte i·record_bytes):
 *   codes : b_m·d/8 bytes.  Code j (the centroid index of rotated coordinate j)
 *           occupies bits [j·b_m, (j+1)·b_m) of the record, least significant
 *           bit first; bit k of the record is bit (k mod 8) of byte (k div 8).
 *   signs : d/8 bytes (prod only).  Bit i (same bit order) is 1 iff the QJL
 *           sign of coordinate i of S·r is +1 (sign(0) = +1).
 *   norm  : float32 ‖x‖₂ of the input row («Шаг 0»).
 *   rnorm : float32 ‖r‖₂ of the residual of the unit-norm row (prod only).
 * A zero input row is stored as norm 0, codes 0, signs all +1, rnorm 0.
 * Decode attention expects the K and V rows of a batch ordered [B][Hkv][T_max].
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TQ_OK 0
#define TQ_EINVAL (-1)        /* bad argument value or shape                       */
#define TQ_EUNSUPPORTED (-2)  /* valid but not implemented (e.g. d not in range)   */
#define TQ_EALIGN (-3)        /* pointer or stride not 16-byte aligned             */
#define TQ_ECUDA (-4)         /* CUDA runtime/driver error (message has details)   */
#define TQ_ENOMEM (-5)        /* device allocation failed in tq_init               */
#define TQ_EWORKSPACE (-6)    /* workspace smaller than tq_decode_workspace_bytes  */

/* Codes in a handle's device status word (tq_device_status) other than the
 * 1..99 of an expired pipeline wait. */
#define TQ_STATUS_APPEND_FULL 200  /* an append found its (batch, KV head) slab full */
#define TQ_STATUS_BAD_CHANNEL 201  /* a channel permutation entry was outside [0, d) */

enum { TQ_MSE = 0, TQ_PROD = 1 };
enum { TQ_BF16 = 0, TQ_F32 = 1 };
enum { TQ_ROT_QR = 0, TQ_ROT_HADAMARD = 1 };

typedef struct tq_ctx* tq_handle;

/* Device pointers to the planes of n_rows packed rows (see above).  signs and
 * rnorm are ignored (may be NULL) for an mse handle; codes is ignored when
 * b_m = 0 (prod with b = 1). */
typedef struct {
    uint8_t* codes;
    uint8_t* signs;
    float* norm;
    float* rnorm;
} tq_planes;

/*
 * tq_init — build one quantizer: Π, S, the Lloyd–Max codebook and its decision
 * boundaries, all determined by (d, bits, variant, seed), and upload them to the
 * current CUDA device.
 *   «Шаг 1»: Π = Q·diag(sign(R_ii)) for G = QR, G a d×d matrix of i.i.d. N(0,1)
 *            draws (SplitMix64 stream seed ⊕ 0x5049524F54415445, uniform
 *            (z>>11)·2⁻⁵³, Box–Muller on consecutive pairs, row-major fill).
 *   «QJL»:   S, d×d i.i.d. N(0,1) from the stream seed ⊕ 0x514A4C534B455443
 *            (prod only; independent of Π).
 *   «Шаг 2»: Lloyd–Max codebook with 2^b_m levels for the exact coordinate law
 *            f_X(x) = Γ(d/2)/(√π Γ((d−1)/2))·(1−x²)^((d−3)/2) on [−1, 1];
 *            boundaries are midpoints of neighbouring centroids.
 * d: multiple of 32 in [32, 256].  bits: 1..4 (mse), 1..4 (prod; b = 1 stores
 * signs only).  variant: TQ_MSE or TQ_PROD.  On success *out owns device memory
 * until tq_destroy.  Synchronous (blocks on the uploads).
 */
int tq_init(int d, int bits, int variant, uint64_t seed, tq_handle* out);

/*
 * tq_init_ex — tq_init with a choice of rotation.  rotation = TQ_ROT_QR is
 * tq_init.  rotation = TQ_ROT_HADAMARD replaces «Шаг 1»'s Π by the randomised
 * Walsh–Hadamard rotation the page's community findings (#3) recommend for the
 * MSE stage, with QJL on its own independent S as before:
 *   Π = H_d·diag(σ)/√d,  (H_d)_ji = (−1)^popcount(j AND i)  (natural-order
 *   Sylvester matrix),  σ_i = +1 if the i-th uniform (z>>11)·2⁻⁵³ of the
 *   SplitMix64 stream seed ⊕ 0x5748545349474E53 is below ½, else −1.
 * The Hadamard rotation needs d to be a power of two (32, 64, 128, 256), else
 * TQ_EUNSUPPORTED; any other rotation value is TQ_EINVAL.  The packed planes,
 * codebook, S and every other call are unchanged.
 */
int tq_init_ex(int d, int bits, int variant, int rotation, uint64_t seed, tq_handle* out);

/* Free everything tq_init allocated.  NULL is accepted. */
int tq_destroy(tq_handle h);

/* Record sizes in bytes of the codes and signs planes (0 when absent). */
int tq_row_bytes(tq_handle h, int* code_bytes, int* sign_bytes);

/*
 * Host-only construction of the same parameters tq_init uploads, in float64,
 * without touching any GPU (for inspection and tests).  Arrays are caller-owned:
 * Pi [d·d] row-major (y = Π·x), S [d·d] row-major (may be NULL; ignored for mse),
 * centroids [2^b_m] ascending, bounds [2^b_m − 1] ascending (NULL allowed).
 */
int tq_build_params_host(int d, int bits, int variant, uint64_t seed,
                         double* Pi, double* S, double* centroids, double* bounds);

/* tq_build_params_host with a rotation argument (as in tq_init_ex). */
int tq_build_params_host_ex(int d, int bits, int variant, int rotation, uint64_t seed,
                            double* Pi, double* S, double* centroids, double* bounds);

/* Host copies of a handle's float64 parameters (same layout as above). */
int tq_get_params(tq_handle h, double* Pi, double* S, double* centroids, double* bounds);

/*
 * tq_quantize — quantize n_rows rows of x into the packed planes.
 * «Шаг 0»–«Шаг 2» (mse); «Собственно TurboQuant» for prod.  Per row x:
 *   norm = ‖x‖₂;  y = Π·x;  code_j = #{k : t_k·norm < y_j} (ties → lower code);
 *   prod: e = y/norm − c[code] (the residual r = Πᵀe in the rotated frame),
 *         rnorm = ‖e‖₂, sign bit i = [(S·r)_i ≥ 0] computed as (S·Πᵀ·e)_i.
 * x: device pointer to n_rows rows of d elements of x_dtype (TQ_BF16 or
 *    TQ_F32), row i starting x_row_stride elements after row i−1
 *    (x_row_stride ≥ d; x_row_stride·element size a multiple of 16 bytes).
 * out: planes with room for n_rows records.  n_rows = 0 is a no-op.
 */
int tq_quantize(tq_handle h, const void* x, int x_dtype, int64_t n_rows,
                int64_t x_row_stride, tq_planes out, void* stream);

/*
 * tq_quantize_kv — tq_quantize(hk, k, …, k_out) and tq_quantize(hv, v, …, v_out)
 * in one call: the key and value rows of a decode step or a prefill chunk (the
 * «KV-кэш» use of the method: K and V are quantized independently, each with
 * its own handle).  Results are bit-identical to the two separate calls.  When
 * both handles are mse with the same d ∈ {64, 128}, b and rotation kind, and
 * the rows are bf16 or fp32, both sides run in ONE launch of the tensor-core
 * kernel (its CTAs split between K and V in proportion to their rows);
 * otherwise the call makes the two launches.  Arguments: as tq_quantize for each
 * side (k_rows / v_rows may differ; either may be 0); both sides share x_dtype.
 * k_out and v_out must not overlap each other or the inputs.  Errors: as
 * tq_quantize, checked for both sides before anything is launched.
 */
int tq_quantize_kv(tq_handle hk, tq_handle hv, const void* k, const void* v, int x_dtype,
                   int64_t k_rows, int64_t v_rows, int64_t k_row_stride, int64_t v_row_stride,
                   tq_planes k_out, tq_planes v_out, void* stream);

/*
 * tq_dequantize — Q⁻¹ of «Шаг 2» plus, for prod, the QJL reconstruction:
 *   x̃ = norm·(Πᵀ·c[code] + √(π/2)/d·rnorm·Sᵀ·z),  z_i = ±1 from the sign bits.
 * y: device pointer to n_rows·d contiguous elements of y_dtype (TQ_F32 or
 *    TQ_BF16).
 */
int tq_dequantize(tq_handle h, tq_planes in, int64_t n_rows, void* y, int y_dtype,
                  void* stream);

/*
 * Size in bytes of the device workspace tq_decode_attention needs for these
 * shapes on the current device (the split count depends on the SM count).
 */
int tq_decode_workspace_bytes(tq_handle hk, tq_handle hv, int B, int Hq, int Hkv,
                              int T_max, size_t* bytes);

/*
 * tq_decode_attention — one decode query per (batch, query head) attending over
 * the compressed cache, never materialising dequantized rows:
 *   q′ = Π_k·q, q″ = S_k·q                     (query rotated once)
 *   s_t = scale·norm_t·(⟨q′, c_k[code_t]⟩ + √(π/2)/d·rnorm_t·⟨q″, z_t⟩)
 *        (= scale·⟨q, k̃_t⟩ by the dequantization rule and ⟨q, Sᵀz⟩ = ⟨Sq, z⟩)
 *   p = softmax(s over t < seq_lens[b]);  o = Π_vᵀ·Σ_t p_t·vnorm_t·c_v[code_t]
 *   (values accumulated in the rotated frame; Πᵀ applied once at the end).
 * Query head h reads KV head h / (Hq/Hkv); Hq must be a multiple of Hkv
 * (Hq ≤ 4096).  hk and hv must share d.
 * q: device [B, Hq, d] of q_dtype (TQ_F32 or TQ_BF16), contiguous.
 * kc, vc: planes holding B·Hkv·T_max rows each, ordered [B][Hkv][T_max].
 * seq_lens: device int32 [B], each in [0, T_max]; an empty context gives o = 0.
 * scale: softmax scale; ≤ 0 selects 1/√d.
 * out: device float32 [B, Hq, d].
 * scores_out: NULL, or device float32 [B, Hq, T_max] receiving the pre-softmax
 *    s_t for t < seq_lens[b] (entries past the length are not written).
 * workspace: device buffer of at least tq_decode_workspace_bytes(...) bytes.
 * Rows of a slab past seq_lens[b] (up to T_max) may be read and are masked;
 * nothing past a slab's T_max rows is read.  A staging wait of the d = 128
 * tensor-core kernel that expires records code 30 in hk's status word, and the
 * merging CTA's wait for the split partials code 31 (tq_device_status); the
 * outputs of that call are then undefined.
 * Stream order is kept: at d = 128 the call launches a kernel that zeroes the
 * workspace's merge tickets and then the decode kernel, each as the
 * programmatic dependent of the kernel before it, and the decode reads none of
 * its inputs before every kernel enqueued ahead of the call has completed.  The
 * decode's prologue then overlaps the tail of a library quantize kernel
 * launched just before it; an event or copy enqueued in between, or a kernel
 * that does not release its dependents early, simply ends that overlap.
 */
int tq_decode_attention(tq_handle hk, tq_handle hv, const void* q, int q_dtype,
                        tq_planes kc, tq_planes vc, const int32_t* seq_lens,
                        int B, int Hq, int Hkv, int T_max, float scale,
                        float* out, float* scores_out,
                        void* workspace, size_t ws_bytes, void* stream);

/*
 * Outlier-channel mixed precision (the page's experiments, KV cache: "outlier"
 * channels kept at more bits than the rest, 32 channels at 3 bits and 96 at 2).
 * A row's d channels are split by a device permutation perm (int32 [d]):
 * perm[0..d_o) are the outlier channels, perm[d_o..d) the others, each entry in
 * [0, d) and each channel once.  Each part is an ordinary quantizer handle of its
 * own dimension (ho: d_o channels, hn: d − d_o; both of one variant), so it has
 * its own norm, rotation, codebook and packed planes.  A perm entry outside
 * [0, d) is never dereferenced: it reads or writes channel 0 and the part
 * handle's status word records TQ_STATUS_BAD_CHANNEL.
 */

/*
 * tq_select_outlier_channels — choose the split from the rows to be cached (the
 * page does not say how outliers are found): energy[j] = Σ_rows x_j² in float64
 * (device [d], written), and perm = the d_o channels of largest energy (ties to
 * the lower channel) ascending, then the others ascending (device int32 [d]).
 * x: device [n_rows, d] with row stride x_row_stride elements (x_dtype TQ_BF16
 * or TQ_F32).  d: multiple of 32 in [64, 256]; d_o: multiple of 32 in
 * [32, d − 32].  Energies are accumulated with float64 atomics, so channels
 * whose energies agree to ~1e-15 relative may be ordered either way.
 */
int tq_select_outlier_channels(const void* x, int x_dtype, int64_t n_rows, int64_t x_row_stride, int d,
                               int d_o, double* energy, int32_t* perm, void* stream);

/* Bytes of the scratch buffer that lets tq_mixed_quantize use the tensor cores. */
size_t tq_mixed_quantize_scratch_bytes(void);

/*
 * tq_mixed_quantize — part o of row i (channels perm[0..d_o)) quantized by ho into
 * record i of out_o, part n (channels perm[d_o..d)) by hn into out_n, exactly as
 * tq_quantize would quantize the gathered sub-rows.  x: device [n_rows, d], row
 * stride x_row_stride ≥ d elements (stride·element size a multiple of 16 bytes).
 * scratch: NULL, or a caller-owned device buffer of scratch_bytes bytes, 256-byte
 * aligned.  With at least tq_mixed_quantize_scratch_bytes() of it, bf16 rows,
 * mse parts, d = 128 and d_o ∈ {32, 64} (b_o ≥ b_n), both parts come out of one
 * tensor-core rotation by M = blockdiag(Π_o, Π_n)·P, whose bf16 halves are built
 * in the scratch on `stream`; otherwise a CUDA-core kernel per part gathers the
 * part's channels itself.  The scratch must not be shared by calls that may run
 * concurrently.
 */
int tq_mixed_quantize(tq_handle ho, tq_handle hn, const int32_t* perm, const void* x, int x_dtype,
                      int64_t n_rows, int64_t x_row_stride, tq_planes out_o, tq_planes out_n,
                      void* scratch, size_t scratch_bytes, void* stream);

/*
 * tq_mixed_quantize_kv — the keys k (k_rows rows: parts hko, hkn, split perm_k)
 * and the values v (v_rows rows: hvo, hvn, perm_v) of one decode step in one
 * call, each side's planes written exactly as tq_mixed_quantize writes them.
 * k and v share x_dtype; each has its own row stride (rules as
 * tq_mixed_quantize).  k_rows or v_rows may be 0: that side's pointers are then
 * not read.  When both sides would take the tensor-core path on their own, have
 * the same d_o and the same (b_o, b_n), and scratch holds at least
 * 2·tq_mixed_quantize_scratch_bytes() (keys' operand first, values' second),
 * one launch builds both operands and one launch quantizes both sides (the
 * grid's CTAs divided between them in proportion to their rows); otherwise the
 * sides are quantized one after the other on `stream`, sharing the scratch.
 * Argument errors name the side ("key" / "value"); bad perm entries are
 * recorded in that side's hko / hvo status word.
 */
int tq_mixed_quantize_kv(tq_handle hko, tq_handle hkn, tq_handle hvo, tq_handle hvn,
                         const int32_t* perm_k, const int32_t* perm_v, const void* k, const void* v,
                         int x_dtype, int64_t k_rows, int64_t v_rows, int64_t k_row_stride,
                         int64_t v_row_stride, tq_planes k_out_o, tq_planes k_out_n, tq_planes v_out_o,
                         tq_planes v_out_n, void* scratch, size_t scratch_bytes, void* stream);

/*
 * tq_mixed_dequantize — both parts dequantized (as tq_dequantize) and written to
 * their channels of y: device [n_rows, d] of y_dtype, contiguous.
 */
int tq_mixed_dequantize(tq_handle ho, tq_handle hn, const int32_t* perm, tq_planes in_o, tq_planes in_n,
                        int64_t n_rows, void* y, int y_dtype, void* stream);

/* Workspace bytes tq_mixed_decode_attention needs for these shapes. */
int tq_mixed_decode_workspace_bytes(tq_handle hko, tq_handle hkn, tq_handle hvo, tq_handle hvn, int B,
                                    int Hq, int Hkv, int T_max, size_t* bytes);

/*
 * tq_mixed_decode_attention — tq_decode_attention over mixed-precision keys and
 * values: the score of token t is the sum of its parts' scores,
 *   s_t = scale·Σ_p ‖k_p,t‖(⟨q′_p, c_p[code]⟩ + √(π/2)/d_p·‖r_p,t‖⟨q″_p, z_p,t⟩)
 * with q′_p = Π_p·q[perm_k part p] (= scale·⟨q, k̃_t⟩ of the mixed dequantized
 * key), and the output is Σ_t p_t·ṽ_t with each value part rotated back by its
 * own Πᵀ (+ Sᵀ) once per head and scattered to its channels by perm_v.  Keys
 * (hko, hkn, perm_k) and values (hvo, hvn, perm_v) may split differently but
 * must have the same total d (64..256).  Planes kc_o, kc_n, vc_o, vc_n hold
 * B·Hkv·T_max records each, ordered [B][Hkv][T_max].  Other arguments as
 * tq_decode_attention; bad perm entries are recorded in hko's status word.
 * The split of the page's experiment — d = 128, 32 outlier channels for keys
 * and for values, mse value parts with (b_o, b_n) ∈ {(3, 2), (4, 3), (4, 2)} and
 * key parts of the same bits, both mse or both prod — and T_max % 4 == 0 run on a
 * tensor-core kernel (staging and merge waits record codes 30 and 31 in hko's
 * status word); every other split on CUDA-core kernels.  The workspace size depends on which (the size query
 * answers for the same handles and T_max).
 */
int tq_mixed_decode_attention(tq_handle hko, tq_handle hkn, tq_handle hvo, tq_handle hvn,
                              const int32_t* perm_k, const int32_t* perm_v, const void* q, int q_dtype,
                              tq_planes kc_o, tq_planes kc_n, tq_planes vc_o, tq_planes vc_n,
                              const int32_t* seq_lens, int B, int Hq, int Hkv, int T_max, float scale,
                              float* out, float* scores_out, void* workspace, size_t ws_bytes,
                              void* stream);

/*
 * tq_decode_append_attention — one decode step that first appends the step's
 * new key and value rows to the packed cache, then attends over the cache with
 * them («Шаг 0»–«Шаг 2» and «Собственно TurboQuant» for the new rows, then the
 * same attention as tq_decode_attention).
 * k_new, v_new: device [B, Hkv, d] rows of kv_dtype (TQ_BF16 or TQ_F32),
 *    contiguous.  The row of (b, h) is quantized with hk (resp. hv) into cache
 *    row (b·Hkv + h)·T_max + seq_lens[b], the next free token of its slab.
 * seq_lens: device int32 [B], read and written: on entry the tokens already
 *    cached, on exit one more.  A slab whose length is already T_max (or
 *    negative) is not written and its length is left as it was; hk's status
 *    word then holds TQ_STATUS_APPEND_FULL (read it with tq_device_status).
 * Attention then covers the updated lengths; q, q_dtype, kc, vc, B, Hq, Hkv,
 * T_max, scale, out and the workspace are as in tq_decode_attention.  Launches
 * on `stream`: one append (K and V rows together; its last block to finish
 * updates the lengths and clears the decode's merge tickets), then the decode
 * (at d = 128 as the append's programmatic dependent: its setup overlaps the
 * append, and it reads lengths, planes and tickets only once the append grid
 * has completed).  The append counts its finished blocks in a device word of
 * hk, so calls that share hk must not overlap on the GPU.
 */
int tq_decode_append_attention(tq_handle hk, tq_handle hv, const void* q, int q_dtype,
                               const void* k_new, const void* v_new, int kv_dtype,
                               tq_planes kc, tq_planes vc, int32_t* seq_lens,
                               int B, int Hq, int Hkv, int T_max, float scale, float* out,
                               void* workspace, size_t ws_bytes, void* stream);

/*
 * Read (and, when clear ≠ 0, reset) the handle's device status word.  Kernels
 * never spin without bound: a pipeline wait that exceeds its time limit records
 * a non-zero code (1..99) there and the kernel returns early (its outputs are
 * then undefined); an append into a full slab records TQ_STATUS_APPEND_FULL.
 * 0 means no such event.  Synchronises the calling thread with the device.
 */
int tq_device_status(tq_handle h, int* status, int clear);

/*
 * tq_check_wait_timeout — exercise the timeout path that tq_device_status
 * reports, without faulting or hanging anything.  Enqueues on `stream` one
 * 32-thread block that waits on a shared-memory mbarrier which nothing
 * completes, using the same bounded wait as the quantize pipelines but with a
 * limit of limit_ns nanoseconds (1 ≤ limit_ns ≤ 10⁹, else TQ_EINVAL).  When
 * the limit expires the block stores `code` (1 ≤ code ≤ 1000, else TQ_EINVAL)
 * into the handle's status word and returns.  Asynchronous; read the result
 * with tq_device_status.  No other buffer is touched.
 */
int tq_check_wait_timeout(tq_handle h, int code, uint64_t limit_ns, void* stream);

/*
 * tq_decode_attention_noalloc — the same computation and arguments as
 * tq_decode_attention, minus the workspace.  It is for callers that cannot call
 * cudaMalloc or hand over a buffer: a serving loop whose device memory is wholly
 * pre-reserved by another allocator (a new allocation could fail or stall the
 * stream), or a thin foreign-language binding that holds stream handles but no
 * device allocator.  The paper has no counterpart; this is a deployment variant.
 *
 * Scratch: one file-scope device array of TQ_NOALLOC_WORKSPACE_BYTES (4 MiB),
 * held by every GPU that loads the library until process exit.  Shapes whose
 * tq_decode_workspace_bytes exceeds it are rejected with TQ_EWORKSPACE before any
 * launch.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress with that device current); make that first call before
 * any stream capture.  The call allocates nothing: no cudaMalloc, cudaFree or
 * allocating library routine.
 * Every call on a device shares the one array and it keeps the last call's
 * contents (nothing in it needs clearing: each call writes all it reads).
 * Calls that overlap on the GPU — on different streams, or from several host
 * threads without ordering — race on it and give undefined results; serialise
 * them, e.g. on one stream.
 */
#define TQ_NOALLOC_WORKSPACE_BYTES (4u << 20)
int tq_decode_attention_noalloc(tq_handle hk, tq_handle hv, const void* q, int q_dtype,
                                tq_planes kc, tq_planes vc, const int32_t* seq_lens,
                                int B, int Hq, int Hkv, int T_max, float scale,
                                float* out, float* scores_out, void* stream);

/* Message for the last error on this thread ("" if none). */
const char* tq_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H */
