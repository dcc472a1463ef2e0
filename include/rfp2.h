/*
 * rfp2.h - C ABI of librfp2.so: block-quantized (ROCmFP2, HFP4G32) GEMV and
 * GEMM on one NVIDIA GB300 (sm_103a).
 *
 * Formats (sources named by page title and section):
 *  - ROCmFP2 block: "ROCmFP2 codebook research report", section "01 Storage".
 *    Ten bytes per 32 weights: q0..q7 hold four 2-bit selectors each,
 *    little-endian (weight 4j+i in bits 2i..2i+1 of byte j), then e0 (scale of
 *    weights 0-15) and e1 (weights 16-31).  A matrix W [M, K] is stored as
 *    uint8 [M, K/32, 10]: blocks row-major, rows contiguous, no row header.
 *  - Codebook (section "02 Quantization"): code 00 -> -4, 01 -> -1,
 *    10 -> +1, 11 -> +4.  Weight = codebook[code] * scale.
 *  - UE4M3 scale byte (section "02 Quantization"): E = b >> 3, M = b & 7;
 *    E = 0 -> M * 2^-10, else (8 + M) * 2^(E - 11).  Bytes 0x00..0x7E are
 *    legal; 0x7F and above are invalid.
 *  - Q8_1-style activations (section "03 Runtime" names Q8_1 activations):
 *    per 32 values d = max|a| / 127 (fp32), q = round-half-away(a / d)
 *    clamped to +-127, q = 0 when d == 0.  q int8 [N, K], d fp32 [N, K/32].
 *  - HFP4G32 row: "HFP4" (hipfire.dev), section "Byte layout - HFP4G32":
 *    16-byte header (f16 row_scale_a, f16 row_scale_b = 0, u16 K/32, u8
 *    flags, reserved) then K/32 blocks of (UE8M0 byte, 16 bytes of E2M1
 *    nibbles, element 2b in the low nibble of byte b).  Row bytes
 *    16 + 17*K/32.  Value = row_scale_a * 2^(e - 127) * E2M1[nibble]
 *    (section "Per-row second-level scale (FP16)"); block byte 0xFF is NaN.
 *
 * Conventions for every entry point:
 *  - Pointers are device memory owned by the caller unless the comment says
 *    host.  The library never allocates device memory and never frees the
 *    caller's buffers.  Arrays are row-major and contiguous.
 *  - Calls are asynchronous on `stream` (0 = legacy default stream) and
 *    return after enqueueing.  The return value reports host-side argument
 *    checks and launch errors only; outputs are valid after the stream
 *    reaches the enqueued work.
 *  - `dev_status` (optional, may be NULL) is one int32 in device memory.  A
 *    kernel that detects an error on the device (a routing id out of range, a
 *    bounded wait that ran out) stores the matching rfp2_status code there;
 *    it never clears it.  The caller zeroes it before the call and reads it
 *    after synchronizing.  With NULL, device-detected errors go unreported.
 *  - Inputs and outputs must not overlap.  Weights are assumed to hold only
 *    legal scale bytes (check with rfp2_validate_weights); an illegal byte
 *    gives unspecified values in the affected outputs, never a fault.
 *  - GPU kernels need K % 256 == 0 (so a row of packed weights is a whole
 *    number of 16-byte units); other K return RFP2_EUNSUPPORTED.
 *  - Ordering: by default no kernel reads W (or any other input) before the
 *    work enqueued ahead of it on the stream has completed, so W may be
 *    written by the kernel just before (e.g. rfp2_pack_weights on the same
 *    stream).  rfp2_set_weight_prefetch(1) lets the GEMV kernels start
 *    streaming W while that earlier kernel is still running (programmatic
 *    dependent launch); x, workspaces and outputs are still touched only
 *    after it has completed.  Turn it on only when no kernel that may still
 *    be in flight on the stream writes W (weights loaded once and
 *    synchronized before the decode loop).
 */
#ifndef RFP2_H
#define RFP2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque stream handle: pass a cudaStream_t. */
typedef struct CUstream_st *rfp2_stream_t;

typedef enum {
    RFP2_OK = 0,
    RFP2_EINVAL = 1,        /* null pointer, negative size, bad enum */
    RFP2_ESHAPE = 2,        /* inconsistent or out-of-range sizes */
    RFP2_EALIGN = 3,        /* a pointer is not aligned as documented */
    RFP2_EUNSUPPORTED = 4,  /* valid input outside what the kernels support */
    RFP2_ECUDA = 5,         /* a CUDA runtime call failed */
    RFP2_EBADSCALE = 6,     /* an illegal scale byte was found */
    RFP2_EBADID = 7,        /* a routing id outside [0, E) */
    RFP2_ETIMEOUT = 8,      /* a bounded device wait ran out */
    RFP2_EWORKSPACE = 9     /* workspace missing or too small */
} rfp2_status;

/* Static string naming a status code ("RFP2_OK", ...). */
const char *rfp2_status_str(int status);

/* Library ABI version (major * 100 + minor). */
int rfp2_version(void);

/* Weight prefetch across kernel boundaries (process-wide, default 0 = off;
 * see "Ordering" above).  With 1, rfp2_gemv, rfp2_gemv_q8 and hfp4_gemv may
 * begin reading W before the kernel enqueued just before them on the stream
 * has completed, which hides the weight stream of one call behind the
 * previous one.  Takes effect for calls enqueued after it returns (a CUDA
 * graph keeps the setting it was captured with).  Always returns RFP2_OK. */
rfp2_status rfp2_set_weight_prefetch(int enable);
int rfp2_weight_prefetch(void);

/* Largest batch (activation columns) the GEMV entry points take. */
#define RFP2_MAX_BATCH 8

/* ---------------------------------------------------------------------------
 * Activation quantization (Q8_1-style blocks, "03 Runtime").
 *   x  fp32 [N, K] device, K % 32 == 0 (K % 256 == 0 not required here).
 *   q  int8 [N, K] device (output).  d fp32 [N, K/32] device (output).
 * Errors: EINVAL (null, N or K < 0), ESHAPE (K % 32), ECUDA.
 */
rfp2_status rfp2_quantize_act(const float *x, int64_t N, int64_t K, int8_t *q, float *d,
                              rfp2_stream_t stream);

/* ---------------------------------------------------------------------------
 * ROCmFP2 GEMV on already-quantized activations ("03 Runtime": expand each
 * code byte to four signed int8 lanes, integer dot against Q8_1 activations,
 * int32 sum per 16-weight half, then y += dA * (d0 * S0 + d1 * S1)).
 *   W  uint8 [M, K/32, 10] device, 16-byte aligned.
 *   q  int8 [N, K], d fp32 [N, K/32] device (from rfp2_quantize_act), both
 *      16-byte aligned.
 *   y  fp32 [N, M] device (output), y[n, m] = sum over row m of W times
 *      column n.  1 <= N <= RFP2_MAX_BATCH.  Each weight block is expanded
 *      once and reused for all N columns ("03 Runtime", multi-column reuse).
 * Errors: EINVAL, ESHAPE (N out of range, M or K <= 0), EUNSUPPORTED
 * (K % 256), EALIGN (W, q or d not 16-byte aligned), ECUDA.
 */
rfp2_status rfp2_gemv_q8(const uint8_t *W, int64_t M, int64_t K, const int8_t *q,
                         const float *d, int64_t N, float *y, int32_t *dev_status,
                         rfp2_stream_t stream);

/* Bytes of workspace rfp2_gemv needs for N columns of length K. */
size_t rfp2_gemv_workspace_bytes(int64_t N, int64_t K);

/* ---------------------------------------------------------------------------
 * ROCmFP2 GEMV from fp32 activations ("ROCmFP2 codebook research report",
 * section "03 Runtime"): quantizes x to Q8_1 blocks and runs the int8 dp4a
 * GEMV in one kernel launch for every batch 1 <= N <= 8; int32 sums per
 * 16-weight half, scales applied after the integer sums.  W is read only
 * after the work enqueued before the call has completed, unless
 * rfp2_set_weight_prefetch(1) is in effect (then the kernel starts streaming
 * W early; see "Ordering").
 *   x fp32 [N, K] device; y fp32 [N, M] device; workspace device, at least
 *   rfp2_gemv_workspace_bytes(N, K) bytes, 256-byte aligned; after the call
 *   it holds q int8 [N, K] followed (at offset rounded up to 256) by d.
 * Errors: as rfp2_gemv_q8, plus EWORKSPACE.
 */
rfp2_status rfp2_gemv(const uint8_t *W, int64_t M, int64_t K, const float *x, int64_t N,
                      float *y, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                      rfp2_stream_t stream);

/* ---------------------------------------------------------------------------
 * rfp2_gemv without any device allocation by anyone.  The pages have no
 * counterpart of this call: it exists for callers that cannot allocate device
 * memory (a plugin whose host runtime owns the memory pool, a process under a
 * fixed memory budget, a path that must work after the pool ran out) and so
 * cannot pass rfp2_gemv a workspace.  Same inputs, outputs and result as
 * rfp2_gemv; the quantized activations go to a fixed scratch array inside the
 * library (73,728 bytes of device memory, held on every GPU that loads the
 * library until the process exits).  Limits: N * K <= 65536; larger sizes
 * return RFP2_EWORKSPACE.  Every call looks up the array's device address
 * on the current device (cudaGetSymbolAddress, a host-side query that
 * allocates nothing), then runs two launches: the quantizer into the array
 * and the GEMV on pre-quantized input.  All calls on a device share the
 * array: calls that overlap on the GPU race on it, so the caller serializes
 * them.  Nothing in the array needs clearing; every call overwrites what it
 * uses.
 * Errors: as rfp2_gemv_q8, plus EWORKSPACE (N * K too large).
 */
rfp2_status rfp2_gemv_noalloc(const uint8_t *W, int64_t M, int64_t K, const float *x, int64_t N,
                              float *y, int32_t *dev_status, rfp2_stream_t stream);

/* ---------------------------------------------------------------------------
 * MoE bulk-expert GEMV (MUL_MAT_ID over the routed experts' rows for a few
 * tokens: "HRX on the Radeon iGPU", section "MoE decode and the kernel
 * cache").
 *   W    uint8 [E, M, K/32, 10] device (E experts, each an M x K ROCmFP2
 *        matrix), 16-byte aligned.
 *   ids  int32 [T, top_k] device: the experts of each token.
 *   x    fp32 [T, K] device.
 *   y    fp32 [T, top_k, M] device (output): y[t, j, :] = W[ids[t, j]] x_t.
 *   Each token is quantized once; each touched expert's blocks are expanded
 *   once for all of its tokens.  1 <= T*top_k <= 4096, E <= 65536.
 *   workspace: rfp2_moe_workspace_bytes(T, top_k, K) bytes, 256-byte aligned.
 * An id outside [0, E) is never dereferenced: its output row y[t, j, :] is
 * filled with NaN and RFP2_EBADID is stored to *dev_status.
 * Errors: EINVAL, ESHAPE, EUNSUPPORTED (K % 256), EALIGN, EWORKSPACE, ECUDA.
 */
size_t rfp2_moe_workspace_bytes(int64_t T, int64_t top_k, int64_t K);
rfp2_status rfp2_moe_gemv(const uint8_t *W, int64_t E, int64_t M, int64_t K,
                          const int32_t *ids, int64_t T, int64_t top_k, const float *x,
                          float *y, void *workspace, size_t workspace_bytes,
                          int32_t *dev_status, rfp2_stream_t stream);

/* ---------------------------------------------------------------------------
 * Prefill GEMM on the tensor cores ("ROCmFP2 codebook research report",
 * section "04 Measured evidence": the end-to-end gain comes from prefill).
 * Y[n, m] = sum_k X[n, k] * w[m, k], with w = codebook * scale decoded
 * exactly to bf16 (at most 4 significant bits times a power of two) inside
 * the GEMM kernel, straight into the tensor cores' shared-memory operand
 * stages, and fp32 accumulation in tensor memory.  One launch; no
 * activation quantization on this path.
 *   W  uint8 [M, K/32, 10] device, 16-byte aligned.  X bf16 bits [N, K]
 *   device, 16-byte aligned.  Y fp32 [N, M] device (output), 16-byte aligned.
 *   M % 16 == 0, N >= 1, K % 256 == 0.
 *   workspace: unused (rfp2_gemm_workspace_bytes returns 0; NULL is fine).
 *   The kernel may start while the previous kernel on the stream is still
 *   running and reads X and W only after that kernel has completed.
 * Errors: EINVAL, ESHAPE, EUNSUPPORTED, EALIGN, ECUDA.
 */
size_t rfp2_gemm_workspace_bytes(int64_t M, int64_t K);
rfp2_status rfp2_gemm(const uint8_t *W, int64_t M, int64_t K, const uint16_t *X, int64_t N,
                      float *Y, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                      rfp2_stream_t stream);

/* ---------------------------------------------------------------------------
 * ROCmFP2 GEMV for verify batches (tens to hundreds of tokens): the result of
 * rfp2_gemv (Q8_1-style activations, "ROCmFP2 codebook research report",
 * section "03 Runtime": expand each block once and reuse it for every
 * activation column) computed on the tensor cores.  Each block is decoded
 * once per call and token tile to exact f16 level * scale values inside the
 * GEMM kernel (straight into tensor memory), each token's quantized
 * activations q * dA are scaled by a power of two and split into two f16
 * pieces (relative residual <= 2^-22), and both pieces are multiplied with
 * fp32 accumulation; each output is within about 1e-6 relative of the exact
 * int-path result.
 *   x fp32 [N, K] device, 16-byte aligned, 1 <= N <= 65535; y fp32 [N, M]
 *   device; W 16-byte aligned; workspace device,
 *   rfp2_gemv_batched_workspace_bytes(M, K, N) bytes, 256-byte aligned
 *   (q int8 [N, K], then d fp32 [N, K/32], each at a 256-byte boundary, then
 *   the two activation pieces and the per-token exponents).
 *   The GEMM kernel starts reading W while the call's activation kernels are
 *   still running (every work enqueued earlier on the stream has completed
 *   by then); W must not be written concurrently from another stream.
 * Errors: EINVAL, ESHAPE, EUNSUPPORTED (K % 256, M % 16), EWORKSPACE, EALIGN,
 * ECUDA; a bounded device wait that ran out stores ETIMEOUT in dev_status.
 */
size_t rfp2_gemv_batched_workspace_bytes(int64_t M, int64_t K, int64_t N);
rfp2_status rfp2_gemv_batched(const uint8_t *W, int64_t M, int64_t K, const float *x,
                              int64_t N, float *y, void *workspace, size_t workspace_bytes,
                              int32_t *dev_status, rfp2_stream_t stream);

/* ---------------------------------------------------------------------------
 * HFP4G32 prefill GEMM: Y[n, m] = row_scale_a(m) * sum_k E2M1[c_mk] *
 * 2^(e_mk - 127) * X[n, k] ("HFP4", sections "Element format (OCP E2M1)",
 * "Block scale - UE8M0", "Per-row second-level scale (FP16)" and "Byte
 * layout - HFP4G32"; no activation quantization on this path).  The weights
 * are expanded exactly to bf16 in the workspace (an E2M1 value times a power
 * of two has at most two significant bits; block byte 0xFF gives NaN), the
 * product runs on the tensor cores with fp32 accumulation, and the f16 row
 * scale multiplies each output in fp32.
 *   W uint8 [M, 16 + 17*K/32] device (HFP4G32 rows), 16-byte aligned;
 *   X bf16 bit patterns [N, K] device, 16-byte aligned; Y fp32 [N, M] device,
 *   16-byte aligned; workspace device, hfp4_gemm_workspace_bytes(M, K) bytes,
 *   256-byte aligned (bf16 weights [M, K], then the row scales as fp32).
 * Errors: EINVAL, ESHAPE, EUNSUPPORTED (K % 256, M % 16), EWORKSPACE, EALIGN,
 * ECUDA; a bounded device wait that ran out stores ETIMEOUT in dev_status.
 */
size_t hfp4_gemm_workspace_bytes(int64_t M, int64_t K);
rfp2_status hfp4_gemm(const uint8_t *W, int64_t M, int64_t K, const uint16_t *X, int64_t N,
                      float *Y, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                      rfp2_stream_t stream);

/* ---------------------------------------------------------------------------
 * Block-scaled FP4 (NVFP4) form of the ROCmFP2 prefill GEMM on the FP4 tensor
 * cores ("ROCmFP2 codebook research report", section "02 Quantization": the
 * UE4M3 scale s(b) is half the E4M3FN value of the byte, so codebook * s(b) =
 * (codebook / 2) * E4M3FN(b) with codebook / 2 in {-2, -0.5, 0.5, 2}, all
 * E2M1 values: a ROCmFP2 block is exactly two NVFP4 blocks).
 *
 * rfp2_to_nvfp4: converts packed ROCmFP2 weights W uint8 [M, K/32, 10]
 *   (2-byte aligned) into the NVFP4 image Wnv (16-byte aligned,
 *   rfp2_nvfp4_weight_bytes(M, K) bytes): E2M1 codes uint8 [M, K/2] (element
 *   2j in the low nibble of byte j), then the scale bytes uint8 [M, K/16]
 *   (the ROCmFP2 scale bytes, unchanged).  Exact.  K % 32 == 0.
 *   Errors: EINVAL, ESHAPE, EALIGN, ECUDA.
 *
 * rfp2_gemm_nvfp4: Y fp32 [N, M] = Xq Wnv^T, where Xq is X (bf16 bit
 *   patterns [N, K], 16-byte aligned) quantized per token to NVFP4 (NVIDIA's
 *   published recipe; the pages name NVFP4 only as a reference format): g =
 *   2688 / amax(row), per 16 values a scale byte E4M3(bmax / 6 * g) rounded
 *   to nearest even, elements E2M1 of (x * g) / scale rounded to nearest
 *   even; y = sum(E2M1_w * s_w * E2M1_x * s_x) / g, fp32 accumulation.  The
 *   activation side is not exact: the result differs from the bf16 GEMM by
 *   the FP4 rounding of the activations (a few percent of |y|).
 *   Wnv from rfp2_to_nvfp4; K % 256 == 0; workspace 256-byte aligned of
 *   rfp2_gemm_nvfp4_workspace_bytes(N, K) bytes; after the call it holds the
 *   quantized tokens: codes [N, K/2], then (at an offset rounded up to 256)
 *   scale bytes [N, K/16], then (rounded up to 256) g fp32 [N].
 *   Errors: EINVAL, ESHAPE, EUNSUPPORTED (K % 256), EWORKSPACE, EALIGN, ECUDA;
 *   a bounded device wait that ran out stores ETIMEOUT in dev_status.
 */
size_t rfp2_nvfp4_weight_bytes(int64_t M, int64_t K);
rfp2_status rfp2_to_nvfp4(const uint8_t *W, int64_t M, int64_t K, uint8_t *Wnv,
                          rfp2_stream_t stream);
size_t rfp2_gemm_nvfp4_workspace_bytes(int64_t N, int64_t K);
rfp2_status rfp2_gemm_nvfp4(const uint8_t *Wnv, int64_t M, int64_t K, const uint16_t *X,
                            int64_t N, float *Y, void *workspace, size_t workspace_bytes,
                            int32_t *dev_status, rfp2_stream_t stream);

/* ---------------------------------------------------------------------------
 * HFP4G32 GEMV ("HFP4", sections "Per-row second-level scale (FP16)" and
 * "v1 correctness-anchor inner loop"): y[n, m] = row_scale_a(m) *
 * sum_b 2^(e_b - 127) * sum_i E2M1[c_i] * x[n, i], fp32 activations, fp32
 * accumulation, row scale applied once at the end of the row.
 *   W  uint8 [M, 16 + 17*K/32] device, 16-byte aligned; x fp32 [N, K];
 *   y fp32 [N, M] (output).  1 <= N <= RFP2_MAX_BATCH, K % 512 == 0 (a row
 *   is then a whole number of 16-byte units).
 *   workspace: hfp4_gemv_workspace_bytes(N, K) bytes, 256-byte aligned (the
 *   activations split into two fp16 pieces in tensor-core fragment order).
 * A block byte 0xFF (block NaN) gives NaN in the affected outputs.
 * Errors: EINVAL, ESHAPE, EUNSUPPORTED (K % 512), EALIGN, EWORKSPACE, ECUDA.
 */
size_t hfp4_gemv_workspace_bytes(int64_t N, int64_t K);
rfp2_status hfp4_gemv(const uint8_t *W, int64_t M, int64_t K, const float *x, int64_t N,
                      float *y, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                      rfp2_stream_t stream);

/* ---------------------------------------------------------------------------
 * rfp2_pack_weights with the importance-weighted scale search ("ROCmFP2
 * codebook research report", section "05 Completed experiment": the squared
 * reconstruction error of every candidate scale has each term weighted by
 * importance_k * sqrt(sigma^2 + x_k^2); the page leaves sigma^2 undefined and
 * it is taken as twice the mean of x^2 over the 32-weight block).  Same block,
 * codebook and code rule; only the chosen scale bytes can differ.  Ties keep
 * the smaller byte; a half whose importance is all zero gets byte 0x00.
 *   W fp32 [M, K] device, 16-byte aligned; importance fp32 [K] device, one
 *   finite value >= 0 per input column (e.g. mean squared activation);
 *   out uint8 [M, K/32, 10] device.
 * Errors: EINVAL, ESHAPE (K % 32), EALIGN, ECUDA.
 */
rfp2_status rfp2_pack_weights_weighted(const float *W, int64_t M, int64_t K,
                                       const float *importance, uint8_t *out,
                                       rfp2_stream_t stream);

/* ---------------------------------------------------------------------------
 * Weight packers (offline preparation; "02 Quantization" for ROCmFP2 and
 * "Quantization recipe (HFP4G32)" for HFP4).  Output is bit-identical to the
 * CPU oracle's packers.
 *  rfp2_pack_weights: W fp32 [M, K] (finite, K % 32 == 0) -> out uint8
 *    [M, K/32, 10].  Each 16-weight half tries every legal UE4M3 byte in
 *    ascending order, picks codes by sign and fp32 |x/s| <= 2.5, and keeps
 *    the first byte with the lowest fp64 squared error.  Non-finite inputs
 *    are a contract violation (their blocks get unspecified bytes).
 *  hfp4_pack_weights: W fp32 [M, K] -> out uint8 [M, 16 + 17*K/32]:
 *    row_scale_a = fp16(max|W|/6), smallest block exponent with
 *    block max <= 6 * 2^(e-127), nearest E2M1 code (ties to even mantissa).
 *    Rows whose max|W|/6 overflows fp16 store RFP2_EINVAL to *dev_status.
 * Errors: EINVAL, ESHAPE, ECUDA.
 */
rfp2_status rfp2_pack_weights(const float *W, int64_t M, int64_t K, uint8_t *out,
                              rfp2_stream_t stream);
rfp2_status hfp4_pack_weights(const float *W, int64_t M, int64_t K, uint8_t *out,
                              int32_t *dev_status, rfp2_stream_t stream);

/* Counts scale bytes >= 0x7F in nblocks packed ROCmFP2 blocks: adds the count
 * to *bad_count (device int64, caller zeroes it) and stores RFP2_EBADSCALE
 * to *dev_status (optional) if any was found. */
rfp2_status rfp2_validate_weights(const uint8_t *W, int64_t nblocks, int64_t *bad_count,
                                  int32_t *dev_status, rfp2_stream_t stream);

/* Debug / test: every int32 half sum of the GEMV's integer path,
 * partials[n, m, h] = sum_{i<16} codebook[code(m, 16h+i)] * q[n, 16h+i],
 * int32 [N, M, K/16] device.  Uses the same expansion code as the GEMV. */
rfp2_status rfp2_debug_half_partials(const uint8_t *W, int64_t M, int64_t K, const int8_t *q,
                                     int64_t N, int32_t *partials, rfp2_stream_t stream);

/* Test hook of the failure handling: one thread waits, with the bounded wait
 * every pipeline kernel uses, on an mbarrier that nothing arrives on.  The
 * wait gives up after the library's 2-second limit and the kernel stores
 * RFP2_ETIMEOUT into *dev_status (device int32, required); nothing faults and
 * the context stays usable.  Errors: EINVAL, EALIGN, ECUDA. */
rfp2_status rfp2_debug_wait_timeout(int32_t *dev_status, rfp2_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* RFP2_H */
