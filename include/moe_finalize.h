/*
 * moe_finalize.h -- C ABI of the GB300 (sm_103a) fused MoE finalize library (libmoe_finalize.so).
 *
 * One call computes, for every token t of a decode batch and every hidden index h:
 *
 *   p_r   = round_act( (sum over valid routes k of scale_r[t,k] * gemm2_r[perm_r[t,k], h]) * rsf
 *                      + shared_r[t,h] )                      for each partial r = 0..R-1
 *   S     = round_act( p_0 + p_1 + ... + p_{R-1} )            FP32 sum in rank order
 *   residual_out[t,h] = round_act( S + residual[t,h] )
 *   norm_out[t,h]     = round_act( (x * rstd) * gamma[h] ),   x = residual_out[t,h],
 *                       rstd = 1 / sqrt( sum_h(x^2) / H + eps )
 *   quant_out / sf_out = optional FP8-E4M3 or NVFP4 encoding of norm_out.
 *
 * All sums and products are FP32; round_act is round-to-nearest-even to the activation type.
 * The routed sum is a chain of fused multiply-adds in route order k = 0..K-1 starting from +0.
 *
 * Where this comes from (web pages, cited by title and section):
 *  - flashinfer PR #6631 "perf(comm): gather MoE-finalize routes together and accumulate in FP32",
 *    Description: FP32 routed sum, factor, shared add and rank sum; each rank's finalized row rounded
 *    once; the rank sum rounded once before residual add and RMSNorm; indices and scales of a chunk
 *    of routes loaded before the rows.  Test changes: routes set to -1; top_k 6/8/10.  Benchmark
 *    script: the Python op's arguments (allreduce_in, residual_in, norm_weight,
 *    expanded_idx_to_permuted_idx, norm_out, residual_out, quant_out, scale_out, launch_with_pdl,
 *    eps, shared_expert_output, expert_scale_factor, routed_scaling_factor).
 *  - TensorRT-LLM PR #16778 "MoE: fp32 accumulation in deferred MoEAllReduce finalize", Fix.
 *  - flashinfer PR #6546 (finalizeKernelSmallBatch), Description: one CTA per (token, hidden slice),
 *    128-bit loads, top-K split over thread groups, PDL trigger at start and wait before reading the
 *    GEMM output; review "Wait for the PDL dependency before reading routing metadata".
 *  - flashinfer PR #3385 "feat: MNNVL Allreduce quant fusion and performance optimization": FP8 and
 *    NVFP4 outputs, scale-factor layouts LINEAR and SWIZZLED_128x4 only, ranks summed in the fixed
 *    order 0..world_size-1, tail guard on the hidden size, optional prenormed (residual) output.
 *
 * Here the R tensor-parallel partials are R sets of input tensors resident in this GPU's memory;
 * nothing crosses GPUs.
 *
 * Conventions for every entry point:
 *  - Pointers named "device" must point to memory of the current CUDA device; the caller owns them.
 *    The library never allocates, frees or synchronizes, and keeps no pointer after a call returns.
 *  - Tensors are dense, row-major, with the shapes given; rows of act tensors must start on 16-byte
 *    boundaries (base pointers 16-byte aligned, H a multiple of 8).
 *  - A negative return value is an error detected on the host BEFORE any work is enqueued; nothing
 *    is written in that case.  moe_finalize_last_error() gives a message for the calling thread.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream) and runs
 *    asynchronously; device-side faults surface at the caller's next synchronization.
 */
#ifndef MOE_FINALIZE_H_
#define MOE_FINALIZE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t == struct CUstream_st* */

#define MFR_ABI_VERSION 2
#define MFR_MAX_PARTIALS 8 /* R */
#define MFR_MAX_TOP_K 64   /* K; the small-batch kernel of flashinfer PR #6546 takes 4 < topK <= 64 */
#define MFR_MAX_HIDDEN 32768

/* Element types. */
typedef enum { MFR_BF16 = 0, MFR_FP16 = 1, MFR_FP32 = 2 } mfr_dtype;

/* Output quantisation (flashinfer PR #3385: FP8 and NVFP4 quantised outputs). */
typedef enum {
  MFR_QUANT_NONE = 0,
  MFR_QUANT_FP8_E4M3 = 1, /* quant_out[t,h] = e4m3_satfinite(norm_out[t,h] * quant_scale)            */
  MFR_QUANT_NVFP4 = 2     /* per 16-element block: sf = e4m3((amax/6) * g), code = e2m1(v * g/sf)    */
} mfr_quant;

/* NVFP4 block-scale layouts (flashinfer PR #3385 review: only LINEAR and SWIZZLED_128x4 accepted). */
typedef enum {
  MFR_SF_ROW_MAJOR = 0,      /* [T, H/16] bytes                                                     */
  MFR_SF_SWIZZLED_128x4 = 1  /* 512-byte tiles of 128 rows x 4 scales; rows padded to 128, the H/16
                                scale columns padded to 4; byte of (m, k) at
                                ((m/128)*ceil(H/64) + k/4)*512 + (m%32)*16 + ((m%128)/32)*4 + k%4    */
} mfr_sf_layout;

/* Kernel choice (MFR_KERNEL_AUTO lets the library pick by batch size). */
typedef enum {
  MFR_KERNEL_AUTO = 0,
  MFR_KERNEL_CLUSTER = 1, /* small batch: one thread-block cluster per token, hidden split over CTAs */
  MFR_KERNEL_STREAM = 2,  /* large batch: persistent CTAs, rows streamed by per-thread async copies */
  MFR_KERNEL_BULK = 3     /* large batch: persistent CTAs, rows staged by bulk copies (cp.async.bulk)
                             that a producer warp issues, several rows per mbarrier-counted stage     */
} mfr_kernel;

/* Flags. */
enum {
  /* Launch with programmatic dependent launch: the kernel lets its dependents launch at its start and
   * waits for the preceding kernel on the stream before reading any input or writing any output. */
  MFR_FLAG_PDL = 1u,
  /* With MFR_FLAG_PDL: perm_idx and expert_scale were complete before the preceding kernel started,
   * so they may be read before the dependency wait (flashinfer PR #6546, PDL ordering item 1).  Do not
   * set it when the kernel right before this one writes the routing. */
  MFR_FLAG_ROUTING_READY = 2u,
  /* Test hook for failure detection: the cluster kernel's exchange barrier expects 4 bytes more than
   * its peers send, so every wait on it runs out after its limit (about 2 s) and is counted by
   * moe_finalize_read_timeouts.  The sums have all landed by then, so the outputs are still complete.
   * It has no effect on plans with one CTA per token or on the stream kernel.  Not for production use. */
  MFR_FLAG_TEST_EXCHANGE_TIMEOUT = 1u << 30,
  /* Test hook for failure detection: the stream kernel's end-of-token barrier (where a group's warps
   * meet to add their sums of squares) expects one arrival more than its warps give, so every wait on
   * it runs out after its limit (about 2 s), is counted by moe_finalize_read_timeouts, and the kernel
   * returns early: tokens past each group's first are then not written, and norm_out and the quantised
   * output of the first are not written either.  No effect on the cluster kernel or in finalize-only
   * mode.  Not for production use. */
  MFR_FLAG_TEST_STREAM_TIMEOUT = 1u << 29
};

/* Status codes. */
enum {
  MFR_OK = 0,
  MFR_ERR_INVALID_ARG = -1, /* a required pointer is NULL, a size is out of range, or misaligned  */
  MFR_ERR_UNSUPPORTED = -2, /* a valid but unsupported combination (dtype, layout, device)        */
  MFR_ERR_CUDA = -3         /* a CUDA runtime call failed while enqueueing (message kept)         */
};

/* One tensor-parallel partial: what one TP rank would hold.  R = 1 is the plain MoE finalize. */
typedef struct {
  const void* gemm2_out;   /* device [num_rows, H] act: permuted GEMM2 output rows                 */
  int64_t num_rows;        /* rows of gemm2_out; a route whose index is outside [0, num_rows) is
                              skipped (-1 marks a masked route)                                     */
  const int32_t* perm_idx; /* device [T, K] int32: expanded route (t, k) -> row of gemm2_out        */
  const void* expert_scale;/* device [T, K] of scale_dtype, or NULL: every scale is 1.0             */
  const void* shared_out;  /* device [T, H] act, or NULL: no shared expert for this partial         */
} mfr_partial;

typedef struct {
  int32_t T;                 /* tokens, >= 0 (0 = nothing to do)                                   */
  int32_t H;                 /* hidden size, multiple of 8 (16 for NVFP4), <= MFR_MAX_HIDDEN        */
  int32_t K;                 /* routes per token (top_k), 1..MFR_MAX_TOP_K                          */
  int32_t R;                 /* partials, 1..MFR_MAX_PARTIALS, summed in order 0..R-1               */
  int32_t act_dtype;         /* mfr_dtype: MFR_BF16 or MFR_FP16                                     */
  int32_t scale_dtype;       /* mfr_dtype of expert_scale: MFR_FP32, MFR_BF16 or MFR_FP16           */
  float routed_scaling_factor; /* multiplies the routed sum (1.0 = off)                            */
  float eps;                 /* RMSNorm epsilon, added to the mean square                           */
  const mfr_partial* partials; /* HOST array of R descriptors, read during the call only            */
  const void* residual;      /* device [T, H] act                                                   */
  const void* gamma;         /* device [H] act: RMSNorm weight                                      */
  void* residual_out;        /* device [T, H] act, or NULL (not written)                           */
  void* norm_out;            /* device [T, H] act, or NULL (not written)                           */
  int32_t quant_mode;        /* mfr_quant                                                           */
  int32_t sf_layout;         /* mfr_sf_layout (NVFP4 only)                                          */
  const float* quant_scale;  /* device fp32 scalar: FP8 encode scale s, or NVFP4 global scale g     */
  void* quant_out;           /* device: FP8 [T, H] bytes (8-byte aligned); NVFP4 [T, H/2] bytes, even
                                element in the low nibble (4-byte aligned).  Required iff
                                quant_mode != NONE                                                  */
  void* sf_out;              /* device NVFP4 block scales (e4m3 bytes), moe_finalize_sf_bytes()
                                bytes; padding bytes are not written.  Required iff NVFP4           */
  uint32_t flags;            /* MFR_FLAG_*                                                          */
  int32_t kernel;            /* mfr_kernel                                                          */
  void* finalize_out;        /* device [T, H] act, or NULL: the finalized MoE output before the
                                residual, S = round(sum over r of p_r) (p_0 when R = 1), the output
                                of the standalone finalize (flashinfer PR #6546, Description:
                                trtllm_moe_run_finalize; TensorRT-LLM PR #16778, Fix: the deferred
                                finalize producer)                                                 */
} mfr_args;

/* Launch geometry chosen for a call (for tests and benchmarks). */
typedef struct {
  int32_t kernel;     /* MFR_KERNEL_CLUSTER, MFR_KERNEL_STREAM or MFR_KERNEL_BULK                    */
  int32_t grid;       /* CTAs launched                                                               */
  int32_t cluster;    /* CTAs per cluster (1 = no cluster)                                           */
  int32_t block;      /* threads per CTA                                                             */
  int32_t smem_bytes; /* dynamic shared memory per CTA                                               */
  int32_t chunk;      /* stream and bulk kernels: hidden elements per pass; cluster kernel: hidden   */
                      /* elements per chunk of a CTA                                                */
  int32_t stages;     /* stream kernel: row slots per group; bulk kernel: stages (each of several    */
                      /* rows); cluster kernel: chunks per CTA                                      */
} mfr_plan;

/* Enqueue the fused finalize.  Returns MFR_OK or a negative status (see above).
 * Required: partials[r].gemm2_out and perm_idx for every r, and at least one of residual_out,
 * norm_out, quant_out, finalize_out.  residual and gamma are required unless finalize_out is the
 * only output (finalize-only mode: no residual add, RMSNorm or quantisation is done and neither is
 * read); gamma is needed also when norm_out is NULL, since the RMS feeds the quantisation.
 * residual_out may be residual itself (the in-place residual update: each element of residual is
 * read by the thread that later writes that element of residual_out).  No other input may overlap an
 * output, and outputs must not overlap each other. */
int moe_finalize_fused(const mfr_args* args, struct CUstream_st* stream);

/* The geometry moe_finalize_fused would use for these arguments on the current device (validates
 * the arguments the same way; enqueues nothing). */
int moe_finalize_plan(const mfr_args* args, mfr_plan* plan);

/* Size in bytes of the NVFP4 block-scale buffer for T x H (flashinfer PR #6631, Test changes: the
 * scale buffer must be sized for the SWIZZLED_128x4 layout; T*H/16 is too small).  <0 on bad input. */
int64_t moe_finalize_sf_bytes(int32_t T, int32_t H, int32_t sf_layout);

/* Size in bytes of quant_out for T x H: T*H (FP8, one E4M3 byte per element), T*H/2 (NVFP4, two E2M1
 * codes per byte), 0 (none) -- the FP8 and NVFP4 quantised outputs of flashinfer PR #3385, Description.
 * <0 on bad input. */
int64_t moe_finalize_quant_bytes(int32_t T, int32_t H, int32_t quant_mode);

/* Static text for a status code (no counterpart on the pages). */
const char* moe_finalize_status_string(int status);

/* Message describing the last error returned to the calling thread ("" if none; no counterpart on
 * the pages). */
const char* moe_finalize_last_error(void);

/* Measurement aid (no counterpart on the pages): enqueue one empty kernel launched the same way as
 * the finalize (1 CTA, with the PDL attribute iff flags has MFR_FLAG_PDL).  Its time in a graph of
 * back-to-back launches is the launch floor the finalize is compared against. */
int moe_finalize_empty_launch(struct CUstream_st* stream, uint32_t flags);

/* Measurement aid (no counterpart on the pages): enqueue one CTA of 32 threads that reads idx[0] (a
 * device int32), then 16 bytes per thread of row idx[0] of `rows` (nrows rows of row_bytes bytes, a
 * device buffer), and writes those 512 bytes to `out` (device, at least 512 bytes): the dependent
 * index -> row -> store chain every finalize begins with, launched like the finalize (PDL attribute
 * iff flags has MFR_FLAG_PDL).  An index outside [0, nrows) writes nothing.  Buffers and row_bytes
 * must be 16-byte aligned and row_bytes >= 512 (else MFR_ERR_INVALID_ARG).  Its time in a graph of
 * back-to-back launches is the latency floor of a gather (launch plus two dependent memory reads). */
int moe_finalize_gather_floor_launch(const int32_t* idx, const void* rows, int64_t nrows, int64_t row_bytes,
                                     void* out, struct CUstream_st* stream, uint32_t flags);

/* Robustness aid (no counterpart on the pages): every wait in the kernels is bounded (about 2 s): the
 * stream kernel's waits on its pipeline barriers and the cluster kernel's wait for its peers' sums of
 * squares.  A wait that runs out records a count on the device and the kernel goes on or returns
 * early.  This reads the count for the current device into *count and resets it.  It synchronizes
 * the device.  A nonzero count means the outputs of some call are incomplete or wrong. */
int moe_finalize_read_timeouts(uint32_t* count);

/* MFR_ABI_VERSION of the loaded library. */
int moe_finalize_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FINALIZE_H_ */
