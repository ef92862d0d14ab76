/*
 * woq.h - C ABI of the weight-only-quantised skinny linear for NVIDIA GB300 (sm_103a).
 *
 * The op ("Doubling LLM token rates in ComfyUI", blog.comfy.org, sections
 * "What is the bottleneck?" and "Optimizing the Linear Kernel"):
 *
 *     y[M x N] = dequant(W[N x K]) . quant8(x[M x K]),   M = 1 .. 8 (int4), 1 .. 4 (int6)
 *
 * W holds 4-bit (W4A8) or 6-bit (W6A8) signed weights with one fp16 scale per
 * row and group of 128 consecutive k; x is quantised per row to int8 with
 * scale amax/127 (round half to even); per group the int8 x int4/int6 dot
 * product is exact in int32, then scaled: term = (d * wscale) * ascale, and
 * y = sum of the terms over the groups (fp32).
 *
 * Conventions for every entry point
 *   - Return value: a woq_status (0 = WOQ_OK).  Arguments are validated on the
 *     host before anything is launched; an invalid call launches nothing and
 *     changes no buffer.  Nothing aborts, traps or waits without a bound.
 *   - "host" pointers are ordinary CPU memory; "device" pointers are CUDA
 *     global memory of the current device.  The caller owns every buffer; the
 *     library allocates no memory (device or pinned) in any entry point.
 *   - Device entry points are asynchronous on the given stream (NULL = the
 *     legacy default stream).  Launch failures return WOQ_ERR_CUDA (the CUDA code
 *     is kept for woq_last_cuda_error); a fault in a kernel surfaces at the
 *     caller's next synchronisation.
 *   - Device buffers must be 16-byte aligned, except y, ascale and dots (4 bytes).
 *   - Empty shapes are valid: M == 0 or N == 0 launches nothing and returns
 *     WOQ_OK; K == 0 (no groups) zero-fills y.
 *   - Weights use the packed device layout written by woq_pack_w4 /
 *     woq_pack_w6 (or their device twins).  Its 256-byte header records
 *     (bits, N, K); kernels check it and, on a mismatch, set a flag in the
 *     workspace status word and leave y untouched.
 *   - Kernels are launched with programmatic dependent launch: a woq kernel may
 *     start streaming weights while the previous kernel in the stream is still
 *     running, and waits for it before it reads activations or touches y or the
 *     workspace.  The weights (and their header) are read before that wait, so
 *     a kernel that writes a launch's weights must not let dependents start
 *     early (griddepcontrol.launch_dependents): ordinary kernels, PyTorch's and
 *     the woq packers included, do not; woq kernels that do never write weights.
 */
#ifndef WOQ_H
#define WOQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define WOQ_API __attribute__((visibility("default")))
#else
#define WOQ_API
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* woq_stream_t;

typedef enum {
  WOQ_OK = 0,
  WOQ_ERR_NULL = 1,      /* a required pointer is NULL */
  WOQ_ERR_ALIGN = 2,     /* a device pointer is not 16-byte aligned */
  WOQ_ERR_SHAPE = 3,     /* M, N, K or bits outside the supported range */
  WOQ_ERR_WORKSPACE = 4, /* workspace smaller than woq_workspace_bytes() */
  WOQ_ERR_LAYOUT = 5,    /* packed buffer size or header does not match (bits, N, K) */
  WOQ_ERR_CUDA = 6,      /* a CUDA runtime call failed (launch, copy, attribute query) */
  WOQ_ERR_DEVICE = 7     /* a kernel reported an error in the workspace status word */
} woq_status;

/* Bits of the workspace status word (see woq_read_status). */
#define WOQ_DEVERR_HEADER 0x1u  /* packed header did not match the call's (bits, N, K) */
#define WOQ_DEVERR_TIMEOUT 0x2u /* a bounded pipeline wait ran out (the kernel gave up) */

/* Library version (major * 10000 + minor * 100 + patch). */
WOQ_API int woq_version(void);

/* Human-readable name of a status code. Never NULL. */
WOQ_API const char* woq_status_string(int status);

/* Largest supported M (activation rows): 8 for int4 weights and act_quant.  int6
 * GEMV / linear launches take M <= 4 (WOQ_ERR_SHAPE above).  int4 launches with
 * M = 5 .. 8 run on the f16 tensor-core consumer (its cost does not grow with M). */
WOQ_API int woq_max_m(void);

/* Largest supported K for a GEMV (fused = 0) or bf16 linear (fused = 1) launch with
 * M activation rows on the current device: the activations stay in shared memory
 * next to at least two ring stages (int8 entry: M * K bytes, M * K <= 98304; bf16
 * entry: 2 * M * K bytes).  0 for invalid arguments. */
WOQ_API int woq_max_k(int bits, int M, int fused);

/* ---------------------------------------------------------------------------
 * Packing (section "Optimizing the Linear Kernel": the GEMV reads weights and
 * group scales from one buffer laid out in its reading order, one contiguous
 * run per thread block).
 *
 * Canonical (checkpoint) layout, the input of the packers:
 *   int4: q4 uint8 [N][K/2]; weight (n, k) is the low nibble of byte k/2 when k
 *         is even and the high nibble when k is odd; two's complement [-8, 7].
 *   int6: q6 uint8 [N][3K/4]; weights 4j .. 4j+3 of a row are the four 6-bit
 *         fields (value i in bits 6i .. 6i+5) of the little-endian 24-bit word
 *         in bytes 3j .. 3j+2; two's complement [-32, 31].
 *   scales: uint16 [N][K/128], fp16 bit patterns, scale of row n, group g.
 * Requirements: N >= 0, K >= 0, K % 128 == 0.
 * Packed layout: a 256-byte header followed by ceil(N/128) * (K/128) blocks, one
 * per (128-row tile, 128-k group), tile-major; each block holds the tile's 128
 * group scales followed by its weights in the order one consumer warp reads
 * them.  Rows beyond N are zero.  The size is woq_packed_bytes(bits, N, K).
 * --------------------------------------------------------------------------- */

/* Bytes of the packed layout for (bits, N, K); 0 if the shape is invalid. */
WOQ_API size_t woq_packed_bytes(int bits, int N, int K);

/* Host -> host.  dst must hold woq_packed_bytes(4, N, K) bytes. Synchronous. */
WOQ_API int woq_pack_w4(const uint8_t* q4, const uint16_t* scales_f16, int N, int K, void* dst, size_t dst_bytes);

/* Host -> host.  dst must hold woq_packed_bytes(6, N, K) bytes. Synchronous. */
WOQ_API int woq_pack_w6(const uint8_t* q6, const uint16_t* scales_f16, int N, int K, void* dst, size_t dst_bytes);

/* Host -> host inverse of the packers: packed bytes back to the canonical layout
 * (q: N * row bytes, scales: N * K/128).  Checks the header. Synchronous. */
WOQ_API int woq_unpack(int bits, const void* packed, size_t packed_bytes, int N, int K, uint8_t* q, uint16_t* scales_f16);

/* Device -> device twin of woq_pack_w4 / woq_pack_w6 (bits = 4 or 6): the
 * canonical weights and scales already sit in device memory; dst is a separate
 * device buffer of woq_packed_bytes(bits, N, K) bytes.  Produces the same bytes
 * as the host packer.  Asynchronous on the stream. */
WOQ_API int woq_pack_device(int bits, const uint8_t* q_dev, const uint16_t* scales_dev, int N, int K, void* dst_dev,
                    size_t dst_bytes, woq_stream_t stream);

/* In-place device relayout ("Doubling LLM token rates in ComfyUI", section
 * "Optimizing the Linear Kernel": the weights are re-laid out in VRAM in place,
 * once per load, with no extra RAM or VRAM).  buf (device, 16-byte aligned, at
 * least woq_packed_bytes(bits, N, K) bytes) holds on entry, from byte 256 on, the
 * canonical weights of all N rows (N * row bytes) directly followed by the
 * canonical fp16 scales (N * K/128 uint16); bytes 0 .. 255 and everything after
 * the scales are scratch.  On return buf holds exactly what woq_pack_device
 * would have written.  No device or host memory is allocated (bytes 0 .. 255
 * serve as the kernel's barrier words until the header is written last).
 * Synchronous: waits for the stream, then reads the header back.  Errors:
 * WOQ_ERR_NULL, WOQ_ERR_ALIGN, WOQ_ERR_LAYOUT (buf_bytes too small), WOQ_ERR_SHAPE
 * (bad shape, or more group scales than the SMs' shared memory can stage:
 * about 16 million on a 152-SM GPU), WOQ_ERR_CUDA (cooperative launch unsupported or failed), WOQ_ERR_DEVICE
 * (a barrier wait ran out: the contents of buf are then undefined and its header
 * invalid, so no GEMV accepts it). */
WOQ_API int woq_relayout_inplace(int bits, void* buf, size_t buf_bytes, int N, int K, woq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Workspace.  GEMV / linear launches split the weight stream evenly over the
 * GPU's SMs; a 128-row tile that straddles CTAs is finished by one of them,
 * which sums the others' partial results (tagged words in the workspace) in a
 * fixed order.  The workspace (device, caller-owned) must be zero-filled once
 * before first use (woq_workspace_init); every successful launch leaves its
 * synchronisation words zero again (after a WOQ_DEVERR_TIMEOUT, zero-fill it
 * again).  Its last M * K * 2 bytes are scratch rows of the SwiGLU entries,
 * overwritten by every such launch (the other entries do not touch them, and
 * accept a workspace without them).  One workspace must
 * not be used by two launches that can run at the same time.  Its size depends
 * on the current device's SM count.
 * --------------------------------------------------------------------------- */

/* Bytes of workspace a GEMV / linear launch of this shape needs on the current device (0 if invalid). */
WOQ_API size_t woq_workspace_bytes(int bits, int M, int N, int K);

/* Zero-fill a workspace on the stream (cudaMemsetAsync). */
WOQ_API int woq_workspace_init(void* ws_dev, size_t ws_bytes, woq_stream_t stream);

/* Synchronously read (and optionally clear) the workspace status word
 * (WOQ_DEVERR_* bits).  Synchronises the stream. */
WOQ_API int woq_read_status(void* ws_dev, size_t ws_bytes, int clear, uint32_t* status_out, woq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Activation quantisation (section "Optimizing the Linear Kernel": the
 * activation is quantised before the integer linear).
 *   x_bf16: device bf16 [M][K]; q: device int8 [M][K]; ascale: device fp32 [M].
 *   Per row: amax = max |x|, ascale = amax / 127 (IEEE division), q = round half
 *   to even of x / ascale (IEEE division), clamped to [-127, 127]; a zero row
 *   gives ascale 0 and q 0.  0 <= M <= woq_max_m(), K >= 0.  Non-finite x is
 *   outside the domain (results undefined).
 * --------------------------------------------------------------------------- */
WOQ_API int woq_act_quant_int8(const void* x_bf16, int M, int K, int8_t* q, float* ascale, woq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Skinny GEMV from int8 activations (sections "What is the bottleneck?" and
 * "Optimizing the Linear Kernel").
 *   wpacked: device, woq_packed_bytes(bits, N, K) bytes from the packer;
 *   q: device int8 [M][K]; ascale: device fp32 [M] (from woq_act_quant_int8);
 *   y: device fp32 [M][N], row-major, overwritten;
 *   ws: device workspace of woq_workspace_bytes(bits, M, N, K) bytes.
 *   0 <= M <= woq_max_m(); N >= 0; K >= 0, K % 128 == 0; K <= woq_max_k(bits, M, 0)
 *   (the activation tile lives in shared memory for the whole launch).
 * --------------------------------------------------------------------------- */
WOQ_API int woq_w4a8_gemv(const void* wpacked, size_t wpacked_bytes, const int8_t* q, const float* ascale, int M, int N,
                  int K, float* y, void* ws, size_t ws_bytes, woq_stream_t stream);
WOQ_API int woq_w6a8_gemv(const void* wpacked, size_t wpacked_bytes, const int8_t* q, const float* ascale, int M, int N,
                  int K, float* y, void* ws, size_t ws_bytes, woq_stream_t stream);

/* ---------------------------------------------------------------------------
 * The whole linear in one launch from bf16 activations: every CTA quantises x
 * exactly as woq_act_quant_int8 does, then runs the GEMV.  Bit-identical to
 * woq_act_quant_int8 followed by woq_w?a8_gemv.  Same arguments as the GEMV,
 * with x_bf16 (device bf16 [M][K]) in place of q and ascale; K <= woq_max_k(bits, M, 1)
 * (shared memory keeps room for x as bf16; rows that fit registers are read from
 * global memory straight into them, longer rows are copied in).
 * --------------------------------------------------------------------------- */
WOQ_API int woq_w4a8_linear_bf16(const void* wpacked, size_t wpacked_bytes, const void* x_bf16, int M, int N, int K, float* y,
                         void* ws, size_t ws_bytes, woq_stream_t stream);
WOQ_API int woq_w6a8_linear_bf16(const void* wpacked, size_t wpacked_bytes, const void* x_bf16, int M, int N, int K, float* y,
                         void* ws, size_t ws_bytes, woq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Prologue fusions (section "Optimizing the Linear Kernel": the RMSNorm or
 * SwiGLU before a linear is folded into its input quantisation, so the tensor
 * between them never goes to memory).  One launch each; h is
 * formed in shared memory, rounded to bf16, then quantised exactly as
 * woq_act_quant_int8 quantises x.
 *
 * RMSNorm: x_bf16 device bf16 [M][K], gamma_bf16 device bf16 [K] (16-byte
 *   aligned), eps >= 0.  h = bf16(RN(RN(x r) gamma)), r = RN(1 / RN(sqrt(RN(ms +
 *   eps)))), the mean of squares ms formed from the exact squares of the bf16 x,
 *   summed as integers at a per-row fixed point (order independent) and rounded
 *   once: ms = RN(RN(S) / K).  An all-zero row (or one whose largest |x| is below
 *   2^-40) gives h = 0.
 * SwiGLU: gate_up device fp32 [M][2K] (the output of a gate+up linear: gate in
 *   columns 0 .. K-1, up in K .. 2K-1), 16-byte aligned.  h = bf16(RN(RN(g sg) u)),
 *   sg = RN(1 / RN(1 + e)), e = e^-g in fp32 by Cody and Waite's reduction and a
 *   degree-7 Taylor polynomial (fused multiply-adds), scaled by 2^n.
 * Otherwise as woq_w4a8_linear_bf16 (the same bounds on M, N, K; K <=
 * woq_max_k(bits, M, 1)).  Each is bit-identical to its woq_*_act_quant_int8
 * twin below followed by woq_w4a8_gemv / woq_w6a8_gemv.
 * --------------------------------------------------------------------------- */
WOQ_API int woq_w4a8_linear_rmsnorm_bf16(const void* wpacked, size_t wpacked_bytes, const void* x_bf16,
                                         const void* gamma_bf16, float eps, int M, int N, int K, float* y, void* ws,
                                         size_t ws_bytes, woq_stream_t stream);
WOQ_API int woq_w6a8_linear_rmsnorm_bf16(const void* wpacked, size_t wpacked_bytes, const void* x_bf16,
                                         const void* gamma_bf16, float eps, int M, int N, int K, float* y, void* ws,
                                         size_t ws_bytes, woq_stream_t stream);
WOQ_API int woq_w4a8_linear_swiglu_f32(const void* wpacked, size_t wpacked_bytes, const float* gate_up, int M, int N,
                                       int K, float* y, void* ws, size_t ws_bytes, woq_stream_t stream);
WOQ_API int woq_w6a8_linear_swiglu_f32(const void* wpacked, size_t wpacked_bytes, const float* gate_up, int M, int N,
                                       int K, float* y, void* ws, size_t ws_bytes, woq_stream_t stream);

/* Unfused twins: RMSNorm (or SwiGLU) then act_quant, writing q int8 [M][K] and
 * ascale fp32 [M] like woq_act_quant_int8.  K % 8 == 0, 2 K bytes of shared memory
 * per row (K <= 113,664); otherwise as the fused forms. */
WOQ_API int woq_rmsnorm_act_quant_int8(const void* x_bf16, const void* gamma_bf16, float eps, int M, int K, int8_t* q,
                                       float* ascale, woq_stream_t stream);
WOQ_API int woq_swiglu_act_quant_int8(const float* gate_up, int M, int K, int8_t* q, float* ascale,
                                      woq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Allocation-free variant of woq_w4a8_linear_bf16 (the pages have no counterpart:
 * this is a service for callers that cannot allocate device memory, such as
 * plugins inside a host application that owns every device allocation, or loops
 * with a fixed memory budget where a cudaMalloc could synchronise or fail).
 *   Same inputs and outputs as woq_w4a8_linear_bf16, without a workspace: its
 *   scratch is a 2 MiB array built into the library, present on every GPU that
 *   loads it until the process exits.  A launch needs 256 bytes plus 2048 * M
 *   bytes per CTA (grids of up to 255 CTAs at M = 4, 1023 / M CTAs in general; on
 *   a 152-SM GPU every shape with M <= 6); a shape whose launch would need more
 *   returns WOQ_ERR_WORKSPACE before anything is enqueued.
 *   The first call on each device looks up the array's device address (with that
 *   device current) and keeps it for the life of the process; make that first call
 *   before any stream capture.  A device reset (cudaDeviceReset) is not supported
 *   afterwards.  Every call zeroes the split-tile words it uses (an asynchronous
 *   memset on the stream) and then launches the linear; it allocates nothing.  The
 *   array's status word is not zeroed: a device-side error (WOQ_DEVERR_*) stays in
 *   it until woq_noalloc_read_status clears it, and with it y may be stale or
 *   partly written.  All calls share the one array, so calls that can overlap on
 *   the GPU (different streams, or a woq linear/GEMV launch running at the same
 *   time) race and must be avoided.
 * --------------------------------------------------------------------------- */
WOQ_API int woq_w4a8_linear_bf16_noalloc(const void* wpacked, size_t wpacked_bytes, const void* x_bf16, int M, int N,
                                         int K, float* y, woq_stream_t stream);

/* Status word of woq_w4a8_linear_bf16_noalloc's built-in scratch on the current
 * device, like woq_read_status: synchronises the stream, writes the WOQ_DEVERR_*
 * bits of every allocation-free call since the last clear to *status_out (host)
 * and, if clear != 0, zeroes them.  Errors: WOQ_ERR_NULL, WOQ_ERR_CUDA. */
WOQ_API int woq_noalloc_read_status(int clear, uint32_t* status_out, woq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Next-linear prefetch hint (section "What is the bottleneck?": a decode step
 * reads the weights of one linear after another, and the memory bus is only
 * busy in bursts; section "Optimizing the Linear Kernel" counts the gaps
 * between the bursts among the costs of a small kernel).
 *   Tells the next GEMV / linear call made by this thread which linear will run
 *   after it: next_wpacked (device, the packed weights of (bits, N, K), at least
 *   woq_packed_bytes(bits, N, K) bytes).  That call, once its own weight stream has
 *   been issued, brings into L2 the first budget_kb KiB (0 = 64) of the weights
 *   each of the next launch's CTAs will stream first, planned as a launch of the
 *   same entry kind and M.  The next launch then finds them in L2; every weight
 *   byte is still read from HBM once.  A hint only: results are the same with or
 *   without it, and a wrong hint only costs bandwidth.  Each GEMV / linear call
 *   consumes the hint (launched or not); next_wpacked NULL clears it.  The hint is
 *   per host thread; under stream capture it is baked into the captured launch.
 *   Errors: WOQ_ERR_SHAPE (bits not 4 or 6, N < 0, K < 0, K % 128, budget_kb
 *   outside [0, 65536]), WOQ_ERR_ALIGN, WOQ_ERR_LAYOUT (next_wpacked_bytes too small).
 * --------------------------------------------------------------------------- */
WOQ_API int woq_prefetch_next(const void* next_wpacked, size_t next_wpacked_bytes, int bits, int N, int K,
                              int budget_kb);

/* ---------------------------------------------------------------------------
 * Debug: the exact per-group integer dot products the GEMV scales.
 *   dots: device int32 [M][N][K/128]; dots[m][n][g] = sum over k in group g of
 *   w(n, k) * q(m, k).  Same bounds as the GEMV (no workspace).
 * --------------------------------------------------------------------------- */
WOQ_API int woq_debug_group_dots(int bits, const void* wpacked, size_t wpacked_bytes, const int8_t* q, int M, int N, int K,
                         int32_t* dots, woq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Tuning: override the launch table for the following GEMV / linear launches
 * of this process.  ctas_per_sm in {1, 2} (0 = table; one CTA fits an SM, so 2
 * runs the grid in two waves, and the SwiGLU entries, whose grid-wide step needs
 * every CTA resident, keep one per SM), stages in [2, 8]
 * (0 = table), prefetch_kb = weight bytes per CTA kept in flight into L2
 * beyond the shared-memory ring, in KiB (-1 = table, 0 = none).  Not
 * thread-safe; meant for benchmark sweeps.  WOQ_ERR_SHAPE for values out of
 * range.
 * --------------------------------------------------------------------------- */
WOQ_API int woq_tune_override(int ctas_per_sm, int stages, int prefetch_kb);

/* The cudaError_t code of the most recent CUDA runtime call that failed inside the
 * library on this thread (an entry returned WOQ_ERR_CUDA), or 0.  The library
 * clears the runtime's own error state after such a failure, so it does not
 * surface again in a later call. */
WOQ_API int woq_last_cuda_error(void);

/* cudaGetErrorName of a code returned by woq_last_cuda_error (static string). */
WOQ_API const char* woq_cuda_error_name(int code);

/* The launch table's choice for one GEMV / linear launch, worked out on the host
 * without launching anything.
 *   entry: 0 = int8 GEMV (woq_w?a8_gemv), 1 = bf16 or RMSNorm linear, 2 = SwiGLU
 *   linear; sms, smem_max: the device to plan for (SM count, opt-in shared memory
 *   per block in bytes), 0 for either = the current device's value.  The tuning
 *   overrides in force apply.  out (host) is filled on WOQ_OK.
 *   Errors: WOQ_ERR_NULL (out NULL); WOQ_ERR_SHAPE (1 <= M <= woq_max_m() for int4
 *   or 4 for int6, N >= 1, K >= 128, K % 128 == 0, M * K <= 98304 and entry in
 *   0..2 not met, or no ring of two stages fits smem_max); WOQ_ERR_CUDA (the
 *   current device could not be queried). */
typedef struct {
  int ctas;            /* grid: one CTA per SM (two with the tuning override), fewer
                          when the matrix has fewer four-block stages than that */
  int stages;          /* shared-memory ring stages (four blocks each) */
  int prefetch_stages; /* stages kept in flight into L2 beyond the ring */
  int smem_bytes;      /* dynamic shared memory per CTA */
  int consumer;        /* 0 = dp4a, 1 = f16 tensor-core MMA */
} woq_launch_plan;
WOQ_API int woq_plan_launch(int bits, int M, int N, int K, int entry, int sms, int smem_max, woq_launch_plan* out);

/* Tests of the bounded waits (the pages describe no failure handling; every wait of a woq
 * kernel on another CTA is bounded so that a stuck CTA never hangs a shared GPU).  Injects one fault into the following launches of this
 * process, made by CTA `cta` (a block index), and bounds the waits it makes run out by
 * wait_limit_us microseconds (0 = the default, 2 s):
 *   kind 1: GEMV / linear launches - that CTA never publishes its split-tile partial
 *           sums; the combiner of such a tile gives up, sets WOQ_DEVERR_TIMEOUT and
 *           leaves that tile's rows of y untouched;
 *   kind 2: SwiGLU linears - that CTA (one of the first half of the grid, the CTAs that
 *           form the row maxima) never counts itself in; every CTA gives up, sets
 *           WOQ_DEVERR_TIMEOUT and leaves y untouched;
 *   kind 3: woq_relayout_inplace - that CTA leaves before the first grid barrier; the
 *           others give up and the call returns WOQ_ERR_DEVICE (buffer contents undefined);
 *   kind 0: no fault (the default).
 * Nothing faults or waits without a bound; after kinds 1 and 2 the workspace must be
 * zero-filled again (woq_workspace_init).  Not thread-safe; for tests only.
 * WOQ_ERR_SHAPE for kind outside 0..3, cta < 0 or wait_limit_us outside [0, 2e6]. */
WOQ_API int woq_tune_fault(int kind, int cta, int wait_limit_us);

/* Tuning: which consumer the following int4 GEMV / linear launches of this process
 * use: 0 = launch table (dp4a), 1 = dp4a, 2 = f16 tensor-core MMA.  Both form the
 * same exact per-group integer dots; outputs agree within the GEMV tolerance.
 * int6 launches always use dp4a.  Not thread-safe; meant for benchmarks and
 * tests.  WOQ_ERR_SHAPE for other values. */
WOQ_API int woq_tune_path(int path);

#ifdef __cplusplus
}
#endif

#endif /* WOQ_H */
