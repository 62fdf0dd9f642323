/*
 * petit.h -- C ABI of the GB300 (sm_103a) BF16-activation x FP4-weight GEMM.
 *
 * The operation (Petit blog "AMD GPU 上 FP4 混合精度推理优化", sections
 * "Introduction" and "Efficient dequantization via preprocessing"; Petit PyPI
 * page, "Features"):
 *
 *     C[m, n] = g * sum_k A[m, k] * Wq[n, k]        Wq = code * block_scale
 *
 *   A   BF16 activations, row-major [m][k].
 *   W   E2M1 (FP4) codes, two per byte, row-major [n][k/2]; element 2j of a
 *       row sits in the low nibble of byte j ("FP4 GEMM on Rubin/Blackwell
 *       with CUTLASS", section 3.3: two FP4 values per byte).
 *   NVFP4: one E4M3 scale per 16 consecutive k of a row, [n][k/16], and an
 *       FP32 per-tensor global scale g (Petit blog, "Detailed performance
 *       analysis": 16 elements share one FP8 scale).
 *   MXFP4: one E8M0 scale per 32 consecutive k, [n][k/32], g = 1 (Petit PyPI
 *       page, "Features").
 *   Accumulation is FP32; C is BF16 (round to nearest even), row-major [m][n].
 *
 * Weights are used through an offline "repack" (Petit PyPI page, "Techniques
 * and performance": weights are shuffled offline, as in Marlin, so the GPU
 * dequantises cheaply).  The repacked buffer holds the codes and the scales
 * (exactly the bytes of both inputs) in an opaque, versioned order
 * (petit_layout_version()).
 *
 * Conventions for every entry point:
 *   - Pointers marked (device) are CUDA device pointers; the caller allocates
 *     and frees them.  The library never allocates or frees memory and never
 *     synchronises, except petit_get_device_status().
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) on the current device.
 *   - Every entry point validates its arguments first; on any error it
 *     returns a non-zero petit_status_t and enqueues nothing.  No entry point
 *     aborts, throws or prints.
 *   - Device pointers must be 16-byte aligned (PETIT_ERR_MISALIGNED).
 *   - Repacked weights are read-only inputs that must not change while GEMMs
 *     that read them are in flight.  Every GEMM kernel is launched with
 *     programmatic dependent launch and starts copying and dequantising its
 *     weights while the kernel before it on the stream is still finishing
 *     (it reads activations and the device global scale, and writes any
 *     output, only after that kernel has completed).  So the kernel enqueued
 *     just before a GEMM on the same stream must not write that GEMM's `rep`
 *     buffer: after copying or modifying weights, synchronise or enqueue
 *     other work before the first GEMM that reads them.  The repack kernels
 *     of this library are the exception: they make their output visible
 *     before they exit, so a GEMM may follow petit_repack_* directly.
 *   - The device must be compute capability 10.3 (GB300, sm_103a)
 *     (PETIT_ERR_ARCH).
 */
#ifndef PETIT_H
#define PETIT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* petit_stream_t; /* same type as cudaStream_t */

typedef enum petit_status {
  PETIT_OK = 0,
  PETIT_ERR_INVALID_ARG = 1,       /* null pointer, bad format id, m < 1 ... */
  PETIT_ERR_UNSUPPORTED_SHAPE = 2, /* n or k not a multiple of 128, too large */
  PETIT_ERR_MISALIGNED = 3,        /* a device pointer not 16-byte aligned */
  PETIT_ERR_WORKSPACE = 4,         /* workspace missing or too small */
  PETIT_ERR_ARCH = 5,              /* current device is not sm_103 */
  PETIT_ERR_CUDA = 6,              /* a CUDA runtime call failed */
  PETIT_ERR_TIMEOUT = 7,           /* a bounded device-side wait ran out */
  PETIT_ERR_BOUNDS = 8             /* an index check failed (bounds-checking build only) */
} petit_status_t;

typedef enum petit_format {
  PETIT_FMT_NVFP4 = 0,     /* E2M1 + E4M3 per 16 + FP32 global scale */
  PETIT_FMT_MXFP4 = 1,     /* E2M1 + E8M0 per 32 */
  PETIT_FMT_NVFP4_F16 = 2  /* NVFP4 repacked for FP16 activations */
} petit_format_t;

/* Version of the repacked weight/scale order.  Stored repacked weights are
 * only valid for the version that wrote them. */
int petit_layout_version(void);

/* Static text for a status code (never NULL). */
const char* petit_status_string(petit_status_t status);

/* ------------------------------------------------------------------ sizes */

/* Bytes of a repacked weight buffer: n*k/2 code bytes plus n*k/16 (NVFP4) or
 * n*k/32 + n*k/1024 (MXFP4: scales and a 16-byte flag field per 128 x 128
 * chunk) bytes; 0 for an unknown format. */
size_t petit_repacked_bytes(int64_t n, int64_t k, int fmt);

/* Bytes of GEMM workspace for this problem on the current device: a device
 * status word, split-tile arrival counters (a fixed 4096-byte region) and
 * FP32 split-K partials.  Returns 0 if the arguments are invalid or no
 * device is usable.  A workspace must be zero-filled once after allocation;
 * every successful GEMM leaves the status word and the counters at zero
 * again (the partials region holds scratch data), so it can be reused by
 * later calls of any shape that fits. */
size_t petit_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k, int fmt);

/* ------------------------------------------------------ offline weight prep */

/* Largest |x| over `count` BF16 values x (device) -> *amax_out (device FP32).
 * Used to derive the NVFP4 global scale.  count >= 1. */
petit_status_t petit_absmax_bf16(const void* x, int64_t count, float* amax_out,
                                 petit_stream_t stream);

/* NVFP4 global scale from the tensor maximum: amax / (6 * 448), in FP32. */
float petit_nvfp4_global_scale(float amax);

/* Quantise BF16 weights W [n][k] (device) to NVFP4: for every row and
 * 16-element block, t = max(amax, 1e-8) / (6 * g) (FP32), scale = E4M3(t)
 * round-to-nearest-even saturating (a zero result becomes 0x01 so scales are
 * positive), codes = nearest E2M1 of x / (scale * g), ties to even, no
 * negative zero.  Block max-abs scaling and the 1e-8 floor follow "FP4 GEMM
 * on Rubin/Blackwell with CUTLASS", sections 2.2 and 5.2.
 * Outputs: w_packed [n][k/2], s_e4m3 [n][k/16] (device).  k % 16 == 0. */
petit_status_t petit_quantize_nvfp4(const void* W, float global_scale,
                                    uint8_t* w_packed, uint8_t* s_e4m3,
                                    int64_t n, int64_t k, petit_stream_t stream);

/* Quantise BF16 weights W [n][k] (device) to MXFP4: per 32-element block the
 * scale is 2^e with e = ceil(log2(max(amax, 1e-8) / 6)) (E8M0 code e + 127,
 * clamped to [0, 254]); codes are the nearest E2M1 of x / 2^e, ties to even.
 * Outputs: w_packed [n][k/2], s_e8m0 [n][k/32] (device).  k % 32 == 0. */
petit_status_t petit_quantize_mxfp4(const void* W, uint8_t* w_packed,
                                    uint8_t* s_e8m0, int64_t n, int64_t k,
                                    petit_stream_t stream);

/* Offline repack (Marlin-style shuffle; Petit blog, "Efficient dequantization
 * via preprocessing"): permutes the packed codes and the scale bytes into the
 * per-tile, per-pipeline-stage order the GEMM streams -- for each 128-row x
 * 128-k chunk, its codes followed by its scales, so one contiguous copy
 * brings both -- with each 32-bit word holding its 8 codes in the bit
 * positions the in-register BF16 decode uses.
 * Inputs w_packed [n][k/2], s_e4m3 [n][k/16] (device, read only); output
 * rep_out of petit_repacked_bytes(n, k, PETIT_FMT_NVFP4) bytes (device, must
 * not overlap the inputs).  n % 128 == 0, k % 128 == 0.
 * Scales must be positive (not 0x00, 0x7F or negative) -- the precondition of
 * Petit's offline transform (Petit PyPI page, "Known limitations"); the
 * library does not check them.  Negative-zero codes are harmless here (they
 * decode to -0.0). */
petit_status_t petit_repack_nvfp4(const uint8_t* w_packed, const uint8_t* s_e4m3,
                                  uint8_t* rep_out, int64_t n, int64_t k,
                                  petit_stream_t stream);

/* Same as petit_repack_nvfp4, with the codes at the bit positions of the
 * FP16 decode used by petit_gemm_f16_nvfp4; output of
 * petit_repacked_bytes(n, k, PETIT_FMT_NVFP4_F16) bytes. */
petit_status_t petit_repack_nvfp4_f16(const uint8_t* w_packed, const uint8_t* s_e4m3,
                                      uint8_t* rep_out, int64_t n, int64_t k,
                                      petit_stream_t stream);

/* Same as petit_repack_nvfp4 for MXFP4 scales s_e8m0 [n][k/32] (code 0xFF is
 * not a number and must not occur).  Each 128 x 128 chunk also records
 * whether all its scale codes are at most 128 (scale <= 2, the case for
 * ordinary weights); the GEMM then decodes its codes with one BF16 multiply
 * instead of two.  Output of petit_repacked_bytes(n, k, PETIT_FMT_MXFP4). */
petit_status_t petit_repack_mxfp4(const uint8_t* w_packed, const uint8_t* s_e8m0,
                                  uint8_t* rep_out, int64_t n, int64_t k,
                                  petit_stream_t stream);

/* Test hook: dequantise repacked weights with the GEMM's own device decode
 * routine and write Wq = code * block_scale as BF16, row-major [n][k]
 * (device).  The global scale is not applied.  Wq is exactly representable,
 * so the result is bit-exact.  (The per-block dump suggested as a debugging
 * aid in "FP4 GEMM on Rubin/Blackwell with CUTLASS", section 7.) */
petit_status_t petit_dequant_bf16(const uint8_t* rep, int fmt, void* W_out,
                                  int64_t n, int64_t k, petit_stream_t stream);

/* Test hook for the FP16 layout: repacked NVFP4 (from petit_repack_nvfp4_f16)
 * -> FP16 Wq [n][k] (device), through the FP16 register decode, bit-exact.
 * n % 128 == 0, k % 128 == 0. */
petit_status_t petit_dequant_f16(const uint8_t* rep, void* W_out, int64_t n, int64_t k,
                                 petit_stream_t stream);

/* --------------------------------------------------------------- the GEMM */

/* C[m][n] = bf16(g * sum_k A[m][k] * Wq[n][k]) with FP32 accumulation.
 * A: BF16 [m][k] (device); rep: repacked NVFP4 weights and E4M3 scales
 * (device); C: BF16 [m][n] (device, must not overlap A);
 * workspace: at least petit_gemm_workspace_bytes(m, n, k, PETIT_FMT_NVFP4)
 * zero-filled bytes (device).  m >= 1 (any value); n % 128 == 0;
 * k % 128 == 0.  Calls that share a workspace must not run concurrently.
 * Device-side waits are bounded: if one runs out, the kernel stops early,
 * C is not valid, and petit_get_device_status() reports PETIT_ERR_TIMEOUT. */
petit_status_t petit_gemm_bf16_nvfp4(const void* A, const uint8_t* rep,
                                     float global_scale, void* C,
                                     int64_t m, int64_t n, int64_t k,
                                     void* workspace, size_t workspace_bytes,
                                     petit_stream_t stream);

/* Same as petit_gemm_bf16_nvfp4, with the global scale g read from device
 * memory: `global_scale_dev` points to one FP32 value (4-byte aligned) that
 * the kernel reads after the preceding kernel on `stream` has completed, so a
 * kernel earlier in the same stream or CUDA graph may compute it (for
 * example from petit_absmax_bf16 output), and a captured graph picks up a new
 * value on every replay without re-capture.  The pages leave g to a host
 * float; this entry point is for serving steps built as CUDA graphs (Petit
 * PyPI page, "Features": integration with serving stacks).  The value must be positive
 * and finite; it is not checked on the device.
 * Errors: as petit_gemm_bf16_nvfp4, and PETIT_ERR_INVALID_ARG for a null or
 * misaligned global_scale_dev. */
petit_status_t petit_gemm_bf16_nvfp4_dscale(const void* A, const uint8_t* rep,
                                            const float* global_scale_dev, void* C,
                                            int64_t m, int64_t n, int64_t k,
                                            void* workspace, size_t workspace_bytes,
                                            petit_stream_t stream);

/* FP16-activation variant (Petit blog, "Introduction": FP16/BF16 activations
 * with FP4 weights): C[m][n] FP16 = g * A[m][k] (FP16) * Wq[n][k]^T, FP32
 * accumulation, FP16 round-to-nearest-even output.  `rep` comes from
 * petit_repack_nvfp4_f16 (the same codes and E4M3 scales as the BF16 path,
 * packed at FP16 bit positions).  Code x E4M3 scale is exact in FP16 for
 * every code and scale, so the dequantised operand equals Wq.  Arguments,
 * workspace (petit_gemm_workspace_bytes(m, n, k, PETIT_FMT_NVFP4_F16)) and
 * errors as petit_gemm_bf16_nvfp4; A and C are FP16 [m][k] and [m][n]. */
petit_status_t petit_gemm_f16_nvfp4(const void* A, const uint8_t* rep, float global_scale,
                                    void* C, int64_t m, int64_t n, int64_t k,
                                    void* workspace, size_t workspace_bytes,
                                    petit_stream_t stream);

/* Same with repacked MXFP4 weights and E8M0 scales (no global scale). */
petit_status_t petit_gemm_bf16_mxfp4(const void* A, const uint8_t* rep, void* C,
                                     int64_t m, int64_t n, int64_t k,
                                     void* workspace, size_t workspace_bytes,
                                     petit_stream_t stream);

/* --------------------------------------------------- MoE grouped GEMM */

/* Mixture-of-experts layer GEMM (Petit PyPI page, "Features": fused MoE
 * kernels for BF16 x MXFP4): num_experts GEMMs that share n and k in one
 * launch, stream-K balanced over all of them.  Expert e multiplies the
 * activation rows [off[e], off[e+1]) of A (BF16 [T][k], T = off[E]; the
 * caller groups the routed tokens by expert) by its own weights and writes
 * the same rows of C (BF16 [T][n]):
 *   C[r][:] = g_e * A[r][:] . Wq_e^T,   off[e] <= r < off[e+1].
 * rep holds the experts' repacked weights back to back, each
 * petit_repacked_bytes(n, k, fmt) bytes (petit_repack_mxfp4 / _nvfp4 output).
 * expert_offsets: host array of num_experts + 1 values, off[0] = 0,
 * non-decreasing (empty experts allowed); 1 <= num_experts <= 64.
 * global_scales (NVFP4 only): host array of num_experts positive floats.
 * workspace: at least petit_moe_workspace_bytes(...) bytes, as for
 * petit_gemm_bf16_nvfp4.  T = 0 is a no-op.  Errors: INVALID_ARG (offsets
 * or scales), UNSUPPORTED_SHAPE (more than 64 experts, n or k not multiples
 * of 128), MISALIGNED, WORKSPACE, ARCH, CUDA. */
size_t petit_moe_workspace_bytes(const int64_t* expert_offsets, int64_t num_experts, int64_t n,
                                 int64_t k, int fmt);
petit_status_t petit_moe_gemm_bf16_mxfp4(const void* A, const uint8_t* rep,
                                         const int64_t* expert_offsets, int64_t num_experts,
                                         void* C, int64_t n, int64_t k, void* workspace,
                                         size_t workspace_bytes, petit_stream_t stream);
petit_status_t petit_moe_gemm_bf16_nvfp4(const void* A, const uint8_t* rep,
                                         const float* global_scales, const int64_t* expert_offsets,
                                         int64_t num_experts, void* C, int64_t n, int64_t k,
                                         void* workspace, size_t workspace_bytes,
                                         petit_stream_t stream);

/* NVFP4 GEMM without a workspace argument.  The pages have no counterpart to
 * this entry point; it is for callers that cannot allocate device memory at
 * the time they call the GEMM: plug-ins whose host framework owns all device
 * memory and forbids allocation inside their enqueue call, and
 * latency-critical loops that cannot afford cudaMalloc's implicit device
 * synchronisation.  It computes what petit_gemm_bf16_nvfp4 computes, but its
 * split-K scratch is an 8 MiB array built into the library's device image:
 * every GPU that loads the library holds those 8 MiB until the process
 * exits, and the call itself allocates and frees nothing.
 *   - The scratch a problem needs is 4352 + 1024 * ctas * bn bytes, where
 *     ctas = min(work units, SMs) and bn is the planner's activation tile
 *     height (16, 32, 64, 128 or 256 for m up to 16, 32, 64, 128, above).
 *     Problems whose scratch exceeds 8 MiB are rejected with
 *     PETIT_ERR_WORKSPACE (use the workspace entry point for them); when the
 *     grid fills all 152 SMs of a GB300, as on the Llama-3-70B shapes, that
 *     accepts m <= 32.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and keeps it for the life of the process; make
 *     that first call before any stream capture.  cudaDeviceReset makes the
 *     kept address stale: do not use this entry point on a device after
 *     resetting it.
 *   - Each call clears the scratch's status word and counters on `stream`
 *     before its kernel.  All calls on a device share the one array, so calls
 *     whose execution overlaps on the GPU (different streams, concurrent
 *     graph branches) race and give wrong results: serialise them.
 *   - Device-side wait time-outs of this variant are not reported (there is
 *     no caller workspace to read them from).
 * Arguments as for petit_gemm_bf16_nvfp4. */
petit_status_t petit_gemm_bf16_nvfp4_noalloc(const void* A, const uint8_t* rep,
                                             float global_scale, void* C,
                                             int64_t m, int64_t n, int64_t k,
                                             petit_stream_t stream);

/* ------------------------------------------------------------------ tuning */

/* Forces the tile shape of every later GEMM plan in this process, for tile
 * tuning and tests (Petit PyPI page, "Known limitations": tile parameters may
 * need tuning for a given matrix size): bn activation rows per tile (the MMA
 * N side: 16, 32, 64, 128 or 256) and ku 128-k chunks per pipeline unit (1,
 * or 2 for bn <= 64; a problem whose k holds an odd number of 128-k chunks
 * runs with 1).  bn = ku = 0 gives the choice back to the planner.  The
 * workspace size queries follow the forced shape, so query them after this
 * call.  Not thread-safe with respect to GEMM calls running concurrently on
 * other host threads.  Errors: PETIT_ERR_INVALID_ARG for any other pair. */
petit_status_t petit_set_tile_config(int bn, int ku);

/* CTA pairs for 128- and 256-row activation tiles.  A single GEMM whose n is
 * a multiple of 256 can run on clusters of two CTAs that take adjacent
 * 128-row weight tiles of the same 256-row work tile; one thread of the pair
 * issues tcgen05 MMAs of M = 256 (cta_group::2) that read both CTAs'
 * dequantised weights, and each CTA holds half of the tile's activation
 * rows, so each SM moves half the activation bytes.  Mode 0 (the default)
 * uses them where the planner expects a gain (256-row tiles, and 128-row
 * tiles of large matrices), mode 1 never, mode 2 wherever they apply (tests
 * and tuning).  Results differ between modes in FP32 summation order only.
 * Not thread-safe with respect to GEMM calls running concurrently on other
 * host threads; query workspace sizes after the call.  Errors:
 * PETIT_ERR_INVALID_ARG for any other mode. */
petit_status_t petit_set_pair_mode(int mode);

/* The plan a GEMM would run with, for tile tuning and for checking the
 * planner without a GPU (Petit PyPI page, "Known limitations": tile
 * parameters may need tuning for a given matrix size).  One launch runs a
 * persistent grid: the output is cut into work tiles of bn activation rows
 * by 128 weight rows (256 with CTA pairs), a tile along k into
 * units_per_tile work units of ku 128-k chunks, and the units, numbered
 * tile by tile with k fastest, into num_ranges consecutive ranges ("stream-K"
 * split: a tile whose units fall into several ranges is summed from their
 * FP32 partials in the workspace). */
typedef struct petit_plan_info {
  int32_t bn;              /* activation rows per tile (the MMA N side) */
  int32_t ku;              /* 128-k chunks per work unit (1 or 2) */
  int32_t cta_pairs;       /* 1: clusters of two CTAs issuing M = 256 MMAs */
  int32_t num_ranges;      /* work ranges: one per CTA, or per CTA pair */
  int32_t num_ctas;        /* CTAs launched (twice num_ranges with CTA pairs) */
  int32_t units_per_tile;  /* work units along k of one tile */
  int64_t num_tiles;       /* work tiles, over all activation tiles and groups */
  int64_t units;           /* num_tiles * units_per_tile */
  uint64_t workspace_bytes; /* workspace the GEMM needs on such a device */
} petit_plan_info_t;

/* Plans C[m, n] = A . Wq^T (arguments as for the GEMM entry points; fmt a
 * petit_format_t) for a device with `num_sms` SMs (1..1024) that holds
 * `pair_capacity` CTA pairs of the pair kernels at once (0..160; 0 plans
 * without CTA pairs), under this process's current petit_set_tile_config and
 * petit_set_pair_mode settings.  No device is touched; on the current
 * device the GEMM runs exactly this plan when num_sms and pair_capacity are
 * petit_device_limits()'s values.  *info receives the plan.  range_starts:
 * NULL, or a host array of max_ranges entries that receives the first unit
 * of every range and then `units` (num_ranges + 1 values, non-decreasing,
 * every range non-empty); when max_ranges is smaller than that, *info is
 * still written and PETIT_ERR_INVALID_ARG is returned.
 * Errors: INVALID_ARG (null info, m < 1, a bad format, num_sms or
 * pair_capacity out of range, range_starts too short), UNSUPPORTED_SHAPE (as
 * for the GEMM). */
petit_status_t petit_plan_gemm(int64_t m, int64_t n, int64_t k, int fmt, int num_sms,
                               int pair_capacity, petit_plan_info_t* info,
                               int64_t* range_starts, int64_t max_ranges);

/* The same for the grouped MoE GEMM (expert_offsets and num_experts as for
 * petit_moe_gemm_bf16_mxfp4; fmt PETIT_FMT_MXFP4 or PETIT_FMT_NVFP4).  No
 * routed tokens (expert_offsets[num_experts] = 0) plans nothing: *info is
 * zeroed and PETIT_OK returned. */
petit_status_t petit_plan_moe(const int64_t* expert_offsets, int64_t num_experts, int64_t n,
                              int64_t k, int fmt, int num_sms, int pair_capacity,
                              petit_plan_info_t* info, int64_t* range_starts,
                              int64_t max_ranges);

/* The current device's SM count and how many CTA pairs of the pair kernels
 * it holds at once (the values the GEMM entry points plan with).  Errors:
 * INVALID_ARG (a null pointer), CUDA (no usable device), ARCH (not sm_103). */
petit_status_t petit_device_limits(int* num_sms, int* pair_capacity);

/* ------------------------------------------------- bounds-checking build */

/* The library also builds as _petit_check.so with every global-memory
 * access, bulk and tensor copy and shared- or tensor-memory buffer index of
 * the GEMM kernel checked against its buffer's extent before use (a debug
 * aid for the illegal-address failures a wrong index or copy coordinate
 * gives: CUTLASS FP4 article, sections 5.1 and 7).  A failed check skips
 * the access, stops the CTA cleanly and records PETIT_ERR_BOUNDS for
 * petit_get_device_status(); no trap, no device assert.  Same API, slower.
 *
 * petit_bounds_checking(): 1 in the bounds-checking build, else 0. */
int petit_bounds_checking(void);

/* Bounds-checking build only: the checks of later GEMM launches in this
 * process use at most `weight_bytes` bytes of each group's repacked weights
 * and `c_elems` elements of C as the extents (a negative value: the true
 * extent), so a test can make a check fail while every access that does
 * happen stays inside its real buffer.  Not thread-safe with respect to
 * concurrent GEMM calls.  The normal build returns PETIT_ERR_INVALID_ARG and
 * changes nothing. */
petit_status_t petit_check_set_limits(int64_t weight_bytes, int64_t c_elems);

/* --------------------------------------------------------- error reporting */

/* Waits for `stream`, then reads the status word the kernels keep at the
 * start of `workspace` (device, workspace_bytes >= 256).  Returns PETIT_OK,
 * PETIT_ERR_TIMEOUT (a bounded wait ran out in some earlier call on this
 * workspace), PETIT_ERR_BOUNDS (in the bounds-checking build of the
 * library, _petit_check.so: a kernel found an index outside its buffer,
 * skipped that access and stopped) or PETIT_ERR_CUDA.  When the word is not
 * zero it is cleared,
 * together with the split-tile arrival counters (bytes 256..4351, when
 * workspace_bytes covers them) that a kernel which stopped early may have
 * left raised; the workspace can then be used again without re-zeroing it.
 * This call synchronises the stream. */
petit_status_t petit_get_device_status(void* workspace, size_t workspace_bytes,
                                       petit_stream_t stream);

/* Fault-detection self test: launches one CTA that waits on a barrier nobody
 * arrives at, with a limit of `timeout_us` microseconds (1..10^6).  The wait
 * runs out, the kernel records PETIT_ERR_TIMEOUT in the workspace status
 * word and returns; the CUDA context stays usable.  workspace_bytes >= 256. */
petit_status_t petit_selftest_timeout(void* workspace, size_t workspace_bytes,
                                      uint32_t timeout_us, petit_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PETIT_H */
