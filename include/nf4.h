/*
 * nf4.h -- C ABI of libnf4, an NF4 weight-only quantized linear layer for one
 * NVIDIA GB300 (sm_103a).
 *
 * The operation comes from the diffuseR pull request "Gemma3 NF4 on GPU:
 * quantized encoder, batch encoding, byte-LUT eager dequant" (#39), Summary
 * paragraph: the seven projection weights of each Gemma3-12B layer are packed
 * to NF4 while activations stay at the compute dtype; the forward dequantizes
 * through a byte lookup table straight into the output buffer and runs a
 * dense matmul.  The page does not print the format; this library fixes it:
 *
 *   - codebook: the 16 NormalFloat-4 values of QLoRA (arXiv:2305.14314,
 *     appendix), ascending, code 7 = 0.0;
 *   - blocks of `block` = 64 consecutive elements of the row-major flattened
 *     weight; one fp32 absmax per block (max |w| over the block), no double
 *     quantization; a partial last block covers the elements it has;
 *   - code = index of the codebook value nearest to w / absmax (fp32 IEEE
 *     division), ties to the lower index; an all-zero block has absmax +0.0
 *     and code 7 everywhere;
 *   - packed byte j holds element 2j in its high nibble and element 2j+1 in
 *     its low nibble;
 *   - dequantized value = bf16_rne( float(bf16_rne(C[code])) * absmax ).
 *
 * The compute dtype (weights, activations, outputs) is bf16 in the plain
 * entry points.  The _ex forms take an nf4_dtype: for fp16 every bf16 above
 * reads binary16 (round to nearest even); for fp32 the dequantized value is
 * C[code] * absmax in fp32 with no further rounding.  The packed format does
 * not depend on the dtype: the same values quantize to the same bytes.
 *
 * bf16 and fp16 tensors cross this interface as 16-bit patterns (uint16_t),
 * fp32 tensors as float.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller (allocate
 *     them however you like; the library never frees them).  The library
 *     itself allocates nothing per call: it keeps, per device, one 4-byte
 *     error word and cached kernel attributes, released when the process
 *     exits.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is stream-ordered and asynchronous: it validates its
 *     arguments on the host, enqueues its kernels and returns.  Nothing
 *     synchronizes except nf4_last_error().
 *   - Argument errors are detected on the host, before anything is enqueued,
 *     and returned as a status; nothing runs on bad input.  A failed launch
 *     returns NF4_ERR_CUDA.  A kernel whose internal wait exceeds its time
 *     limit (about one second) records NF4_ERR_TIMEOUT in the device error word
 *     and exits early; nf4_last_error() reports it.  No call aborts the
 *     process or throws.
 *   - Checked build (compiled with -DNF4_CHECKED; the library's build script
 *     makes it on request, never as the default libnf4.so): every kernel
 *     access to global memory that is not a TMA tensor copy first tests its
 *     index against the extent of the buffer it addresses.  An index outside
 *     skips the access and records NF4_ERR_BOUNDS, which nf4_last_error()
 *     reports; the outputs are then undefined.  On valid arguments the
 *     checked build computes the same bits as the normal one and reports
 *     nothing.  The normal build contains no such test.
 *   - The current CUDA device must be an sm_103 GPU (else NF4_ERR_DEVICE).
 *   - Per device the library resolves, on its first call there, the device
 *     addresses of its own __device__ objects (the error word, and the scratch
 *     array of nf4_linear_noalloc) and caches them for the life of the
 *     process.  A cudaDeviceReset() discards them: do not call the library on
 *     a device after resetting it in the same process.
 */
#ifndef NF4_H_
#define NF4_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NF4_API __attribute__((visibility("default")))
#else
#define NF4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nf4_status {
    NF4_OK = 0,
    NF4_ERR_NULL = 1,       /* a required pointer is NULL */
    NF4_ERR_SHAPE = 2,      /* a size is negative, odd where it must be even, or K % 64 != 0 */
    NF4_ERR_ALIGN = 3,      /* a pointer lacks the alignment the entry point requires */
    NF4_ERR_BLOCKSIZE = 4,  /* block != 64 */
    NF4_ERR_WORKSPACE = 5,  /* workspace NULL or smaller than nf4_linear_workspace_size() */
    NF4_ERR_DEVICE = 6,     /* no current device, or it is not sm_103 */
    NF4_ERR_CUDA = 7,       /* a CUDA runtime call or launch failed */
    NF4_ERR_TIMEOUT = 8,    /* a kernel gave up on a bounded wait (reported by nf4_last_error) */
    NF4_ERR_DTYPE = 9,      /* an nf4_dtype this entry point does not take */
    NF4_ERR_BOUNDS = 10     /* checked build only: a kernel index fell outside its buffer (nf4_last_error) */
} nf4_status;

/* Compute dtypes of the _ex entry points. */
typedef enum nf4_dtype {
    NF4_DTYPE_BF16 = 0,
    NF4_DTYPE_F16 = 1,
    NF4_DTYPE_F32 = 2
} nf4_dtype;

/* The only block size supported. */
#define NF4_BLOCK 64

/*
 * nf4_quantize -- blockwise absmax NF4 quantization of one bf16 tensor.
 * Page: "Gemma3 NF4 on GPU" (#39), Summary: the projection weights are packed
 * to NF4.
 *
 *   w       [numel] bf16 bits, any layout the caller flattens row-major
 *   numel   number of elements; even, >= 0 (0 enqueues nothing)
 *   block   must be NF4_BLOCK
 *   packed  [numel / 2] bytes out
 *   absmax  [ceil(numel / 64)] fp32 out
 *
 * Alignment: none required; 16-byte aligned w and 8-byte aligned packed take
 * the vectorized kernel, anything else a slower element-wise kernel with
 * identical results.  Results are bit-exact: one correct answer exists.
 * Inputs must be finite (NaN/Inf give unspecified codes).
 */
NF4_API nf4_status nf4_quantize(const uint16_t* w, int64_t numel, int32_t block, uint8_t* packed,
                        float* absmax, void* stream);

/*
 * nf4_dequantize -- NF4 to bf16 through a 256-entry byte lookup table.
 * Page: "Gemma3 NF4 on GPU" (#39), Summary: the eager dequant uses a byte LUT,
 * one index per packed byte, gathered straight into the output buffer.
 *
 *   packed  [numel / 2] bytes;  absmax [ceil(numel / 64)] fp32
 *   numel   even, >= 0;  block must be NF4_BLOCK
 *   out     [numel] bf16 bits
 *
 * Alignment: none required; 16-byte aligned out and 4-byte aligned packed take
 * the vectorized kernel.  Bit-exact.
 */
NF4_API nf4_status nf4_dequantize(const uint8_t* packed, const float* absmax, int64_t numel,
                          int32_t block, uint16_t* out, void* stream);

/*
 * nf4_linear -- Y = X . deq(W)^T, the NF4 weight-only linear layer (no bias).
 * Page: "Gemma3 NF4 on GPU" (#39), Summary: ltx23_nf4_linear, the module the
 * loader swaps in for each projection.
 *
 *   x        [M, K] bf16 bits, row-major (row pitch K)
 *   packed   [N, K / 2] bytes and absmax [N, K / 64] fp32: W [N, K] quantized
 *            by nf4_quantize (row-major flattening)
 *   y        [M, N] bf16 bits out, row-major; fp32 accumulation, one bf16
 *            rounding at the end
 *   workspace, workspace_bytes  scratch of at least
 *            nf4_linear_workspace_size(M, N, K) bytes (may be NULL when that
 *            size is 0, i.e. M >= 128).  Its first NF4_WORKSPACE_HEADER_BYTES
 *            bytes are arrival counters of the M <= 16 kernel: they must be
 *            zero before the workspace's first use, and every call -- one
 *            that reports NF4_ERR_TIMEOUT included -- leaves them zero again,
 *            so a workspace zeroed once can be reused for any shape, on one
 *            stream at a time.  The rest needs no initialisation and is
 *            clobbered.
 *
 * Requirements: M, N >= 0, K > 0, K % 64 == 0, block == NF4_BLOCK; x, packed, y
 * and workspace 16-byte aligned, absmax 4-byte aligned.  The weight is the
 * dequantizer's: each element is bf16_rne(float(bf16(C[code])) * absmax) for
 * any fp32 absmax (also one that is not a bf16 value, as from a weight
 * quantized at fp32).  Not bit-exact: the fp32 accumulation order is the
 * kernel's, but repeated calls on the same inputs give the same bits; the
 * result matches an fp64 matmul of the dequantized weights to within bf16
 * output rounding plus fp32 summation error.  Row m of Y depends only on row
 * m of X and on the weight, but the kernel -- and with it the fp32 summation
 * order -- is chosen by the shape, so the same row computed in a call with
 * another M may differ in its last bits.  After NF4_ERR_TIMEOUT (see
 * nf4_last_error) y is undefined.
 */
NF4_API nf4_status nf4_linear(const uint16_t* x, int64_t M, int64_t K, const uint8_t* packed,
                      const float* absmax, int64_t N, int32_t block, uint16_t* y,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * nf4_linear_geglu -- the gate and up projections of a Gemma3 MLP in one
 * fused NF4 GEMM, with the GELU-gated product as its epilogue:
 *   y[m][n] = bf16( gelu_tanh(G[m][n]) * G[m][F + n] ),   G = X . deq(W)^T,
 * gelu_tanh(g) = g/2 * (1 + tanh(sqrt(2/pi) * (g + 0.044715 g^3))) (the tanh
 * form of GELU, Hendrycks and Gimpel, arXiv:1606.08415, section 2).  The
 * diffuseR page "Gemma3 NF4 on GPU" (#39), Summary, quantizes the gate and up
 * projections with the other five; this entry point saves writing both
 * projections' outputs and reading them back for the activation.
 *
 *   x        [M, K] bf16 bits, row-major
 *   packed   [2F, K / 2] bytes and absmax [2F, K / 64] fp32: ONE weight
 *            [2F, K] = the gate weight (rows 0 .. F-1) followed by the up
 *            weight (rows F .. 2F-1), quantized by nf4_quantize as one tensor
 *   F        the MLP's intermediate width (outputs per row)
 *   y        [M, F] bf16 bits out, row-major; G in fp32, the activation and
 *            the product in fp32, one bf16 rounding at the end
 *   workspace, workspace_bytes  at least nf4_linear_workspace_size(M, 2F, K)
 *            bytes (NULL allowed when that is 0), with the zeroed counter
 *            header described at nf4_linear
 *
 * Requirements and errors as for nf4_linear with N = 2F (F < 2^30).  Not
 * bit-exact: matches gelu_tanh(g) * u of an fp64 matmul of the dequantized
 * weights to within fp32 summation error, the fp32 activation and one bf16
 * rounding.
 */
NF4_API nf4_status nf4_linear_geglu(const uint16_t* x, int64_t M, int64_t K, const uint8_t* packed,
                                    const float* absmax, int64_t F, int32_t block, uint16_t* y,
                                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * The same operations at another compute dtype.
 * Page: "Gemma3 NF4 on GPU" (#39), Summary: the tensors that are not
 * quantized stay in the compute dtype, whatever it is.
 *
 * nf4_quantize_ex    w is [numel] of `dtype` (bf16, fp16 or fp32); alignment
 *                    as nf4_quantize with "16-byte aligned w" for the fast
 *                    kernel; w must be aligned to its element size.
 * nf4_dequantize_ex  out is [numel] of `dtype`; fp32 output is
 *                    C[code] * absmax in fp32 (4 bytes per element written).
 * nf4_linear_ex,     x and y of `dtype`:
 * nf4_linear_geglu_ex  - bf16, fp16: the weight operand is exactly
 *                      nf4_dequantize_ex's value of that dtype,
 *                      DT_rne(float(DT(C[code])) * absmax), for any fp32
 *                      absmax (the kernels multiply in one paired 16-bit
 *                      operation when the absmax is itself a DT value, and in
 *                      fp32 with one rounding otherwise -- so an absmax above
 *                      fp16's range gives +-inf weights and 0 for code 7, as
 *                      the dequantizer does); fp32 accumulation, one rounding
 *                      of Y to DT.
 *                    - fp32: runs on the tf32 tensor cores.  The weight is
 *                      C[code] * absmax in fp32 rounded to tf32 (10 fraction
 *                      bits, to nearest, ties away from zero); the tensor
 *                      core reads X's values with their fraction truncated to
 *                      10 bits; fp32 accumulation and fp32 Y, no further
 *                      rounding.  Each product is within 2^-9 relative of
 *                      the exact fp32 one.
 *
 * Results, requirements and errors otherwise as the bf16 forms; a dtype
 * outside nf4_dtype returns NF4_ERR_DTYPE.
 */
NF4_API nf4_status nf4_quantize_ex(const void* w, nf4_dtype dtype, int64_t numel, int32_t block,
                                   uint8_t* packed, float* absmax, void* stream);
NF4_API nf4_status nf4_dequantize_ex(const uint8_t* packed, const float* absmax, int64_t numel,
                                     int32_t block, nf4_dtype dtype, void* out, void* stream);
NF4_API nf4_status nf4_linear_ex(const void* x, nf4_dtype dtype, int64_t M, int64_t K,
                                 const uint8_t* packed, const float* absmax, int64_t N, int32_t block,
                                 void* y, void* workspace, size_t workspace_bytes, void* stream);
NF4_API nf4_status nf4_linear_geglu_ex(const void* x, nf4_dtype dtype, int64_t M, int64_t K,
                                       const uint8_t* packed, const float* absmax, int64_t F,
                                       int32_t block, void* y, void* workspace,
                                       size_t workspace_bytes, void* stream);

/* Bytes of workspace nf4_linear needs for this shape, at any dtype (host
 * only, no device call): 0 for M >= 128, else at least
 * NF4_WORKSPACE_HEADER_BYTES.  Returns NF4_ERR_NULL / NF4_ERR_SHAPE on bad
 * arguments. */
#define NF4_WORKSPACE_HEADER_BYTES 4096
NF4_API nf4_status nf4_linear_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes);

/*
 * nf4_linear_noalloc -- nf4_linear for M < 128 that needs no caller workspace.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory themselves (for example a plugin whose host
 * application owns the whole device memory pool and forbids extensions from
 * allocating, or a path where cudaMalloc's implicit device synchronization is
 * not acceptable).  It computes what nf4_linear computes for the same
 * arguments, with the split-K scratch in a fixed library-owned device array of
 * NF4_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until the
 * process exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *   x, M, K, packed, absmax, N, block, y, stream: as for nf4_linear, M < 128.
 *
 * Errors: M >= 128 -> NF4_ERR_SHAPE (nf4_linear needs no workspace there);
 * a shape whose scratch (nf4_linear_workspace_size) exceeds
 * NF4_NOALLOC_SCRATCH_BYTES -> NF4_ERR_WORKSPACE; otherwise as nf4_linear.
 * The first call on a device resolves the array's device address (one
 * cudaGetSymbolAddress with that device current): make it before any stream
 * capture.  All calls on a device share the array: calls that overlap on the
 * GPU (other streams, other host threads) race and must be serialised by the
 * caller.  Each call clears the array's counter header on its stream (a
 * memset, no allocation) before its kernel; the rest needs no clearing.
 * After NF4_ERR_TIMEOUT y is undefined.
 */
#define NF4_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
NF4_API nf4_status nf4_linear_noalloc(const uint16_t* x, int64_t M, int64_t K, const uint8_t* packed,
                                      const float* absmax, int64_t N, int32_t block, uint16_t* y,
                                      void* stream);

/* Synchronize `stream`, then read and clear this device's error word (the
 * first error any kernel recorded since the last read).  Returns NF4_OK,
 * NF4_ERR_TIMEOUT (a kernel gave up on a wait), NF4_ERR_BOUNDS (checked build:
 * an index outside its buffer), or NF4_ERR_CUDA if the synchronization itself
 * failed. */
NF4_API nf4_status nf4_last_error(void* stream);

/* Static, NUL-terminated name of a status code ("NF4_OK", ...). */
NF4_API const char* nf4_status_string(nf4_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
NF4_API int32_t nf4_version(void);

/* Number of kernels this library has enqueued in this process, on any
 * device or stream (a monotone counter, for accounting and tests). */
NF4_API uint64_t nf4_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* NF4_H_ */
