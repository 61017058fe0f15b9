/*
 * nvfp4_moe.h -- C ABI of the NVFP4 (W4A4) MoE expert forward for GB300 (sm_103a).
 *
 * What the library computes is the expert path described on the page
 * "Gemma 4 NVFP4 MoE 空输出" (taking-lying-flat.github.io, a write-up of vLLM
 * issue #51525), cited below as [page, section / figure]:
 *
 *   token reorder -> a1 quantisation -> grouped w13 GEMM
 *     -> SiLU(gate)*up + a2 quantisation -> grouped w2 GEMM
 *     -> restore token order and sum with the routing weights
 *                                  [page, §矩阵融合 "MoE FFN", pipeline figure]
 *
 * preceded by the check the page says was missing: every expert's stored
 * input-scale slot must be written and finite before its reciprocal is taken
 * [page, ROOT CAUSE].
 *
 * Common rules for every entry point
 *   - Pointers named *_host are host memory; every other pointer is DEVICE
 *     memory on the current CUDA device.  All memory is owned by the caller;
 *     the library allocates no device memory and keeps no per-call state.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     stream-ordered and asynchronous unless the entry point says otherwise.
 *   - The return value is an nvfp4_status.  On any status other than
 *     NVFP4_OK no output buffer has been written, except where noted.
 *     nvfp4_last_error_string() gives a one-line reason (thread-local).
 *   - BF16 tensors are passed as uint16_t bit patterns.
 *   - Shapes: E experts, H hidden size, I expert intermediate size, T tokens,
 *     k experts per token, R = T*k routed rows.  Supported: 1 <= E <= 1024,
 *     1 <= k <= min(32, E), H % 256 == 0, I % 64 == 0 (nvfp4_quantize_experts
 *     alone needs only H % 64 == 0), 0 <= T, R < 2^30.
 *
 * Data formats [page, §NVFP4]
 *   - FP4 E2M1 codes, two per byte: element 2i in the low nibble of byte i,
 *     element 2i+1 in the high nibble.
 *   - One FP8 E4M3 (OCP E4M3FN) block scale per 16 consecutive elements of a
 *     row.  Two scale layouts exist:
 *       NVFP4_SF_LINEAR    [rows, K/16] row-major bytes;
 *       NVFP4_SF_SWIZZLED  the tensor-core layout: the matrix is cut into
 *                          tiles of 128 rows x 64 elements (4 scales per row),
 *                          each stored as 512 contiguous bytes, tiles ordered
 *                          row-tile-major; inside a tile the scale of row r,
 *                          block j sits at byte (r%32)*16 + (r/32)*4 + j.
 *                          Rows are padded to a multiple of 128 and the
 *                          64-element columns to a whole number of tiles; the
 *                          padding holds zero bytes.
 *   - Per-expert FP32 scales are stored in the dequantisation direction, as a
 *     calibration writes them: input_scale (activations) and weight_scale_2
 *     (weights).  The quantiser's global scale is their FP32 reciprocal.
 */
#ifndef NVFP4_MOE_H
#define NVFP4_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *nvfp4_stream_t; /* identical to cudaStream_t */

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,         /* null pointer, bad shape, id outside [0, E) */
    NVFP4_ERR_SCALE_INVALID = 2,       /* an input / weight scale slot failed validation */
    NVFP4_ERR_UNSUPPORTED_SHAPE = 3,   /* shape outside the supported set above */
    NVFP4_ERR_CUDA = 4,                /* a CUDA runtime / driver call failed */
    NVFP4_ERR_DEVICE_TIMEOUT = 5,      /* a bounded device-side wait expired */
    NVFP4_ERR_WORKSPACE_TOO_SMALL = 6, /* ws_bytes below the size query's answer */
    NVFP4_ERR_SCALE_RANGE = 7,         /* reserved; no entry point returns it (UE8M0 scales are carried
                                          per row, see NVFP4_UE8M0_SCALES) */
} nvfp4_status;

enum { NVFP4_SF_LINEAR = 0, NVFP4_SF_SWIZZLED = 1 };

/* Block-scale format of a weight set (nvfp4_prepare_weights_format). */
enum { NVFP4_SF_E4M3 = 0 };

/* OR'ed into a quantiser's scale layout (or passed as sf_format): block scales
 * as UE8M0 bytes instead of E4M3 [page "Gemma 4 NVFP4 MoE 空输出", MoE section:
 * the quantiser template's UE8M0_SF flag].  A UE8M0 byte b is the power of
 * two 2^(b - 127) (255 is NaN, never written).  The scale of a block is the
 * E4M3 path's t = fl(fl(g*amax)/6) rounded up to a power of two, clamped to
 * 2^-127 .. 2^127, so no element of the block saturates; the codes are then
 * e2m1(fl(fl(x*g)/s)) as in the E4M3 path.  nvfp4_moe_forward runs with
 * UE8M0 block scales throughout under NVFP4_UE8M0_SCALES. */
enum { NVFP4_SF_UE8M0 = 4 };

/* Element type of the router's logits (nvfp4_router_topk). */
enum { NVFP4_LOGITS_F32 = 0, NVFP4_LOGITS_BF16 = 1 };

/* Flags of nvfp4_moe_forward / nvfp4_moe_forward_host. */
enum {
    /* Skip the synchronous host check of the scales.  The device still
     * validates them, and on a bad slot every later kernel of the call exits
     * without writing; nvfp4_moe_status() then reports NVFP4_ERR_SCALE_INVALID. */
    NVFP4_SCALES_PREVALIDATED = 1u,
    /* Synchronise at the end of the call and report device-side errors
     * (a bad scale slot or an expired wait) in the return value. */
    NVFP4_SYNC_CHECK = 2u,
    /* The UE8M0 variant [page "Gemma 4 NVFP4 MoE 空输出", MoE section: the
     * quantiser's UE8M0_SF flag]: the weights carry UE8M0 block scales (from
     * nvfp4_quantize_weights_format, prepared with nvfp4_prepare_weights_format
     * and NVFP4_SF_UE8M0), and both activation quantisations take UE8M0 scales
     * (see NVFP4_SF_UE8M0); every other step is unchanged.  The block-scaled
     * FP4 tensor-core MMA is fed E4M3 scale bytes, whose normal powers of two
     * span 15 binades (2^-6 .. 2^8), so each GEMM operand row -- a row of
     * activations, or the weight row of one output column -- carries its
     * UE8M0 scales relative to its own largest one: that largest scale
     * travels as 2^8, the others as the same power of two below it, and the
     * epilogue multiplies the row's power of two back (an exact product, per
     * activation row and per output column).  Any scale in the UE8M0 range is
     * accepted, whatever the calibration.  A block whose scale is more than
     * 14 binades below the largest of its own row contributes zero (its
     * values are below 2^-14 of that row's largest block).  The intermediates
     * (sf1, sf2 of nvfp4_moe_intermediates_of) hold the UE8M0 bytes.  The
     * prepared weights must match the flag (else NVFP4_ERR_INVALID_ARG on the
     * device, nothing written).  Not accepted by nvfp4_moe_forward_w4a16. */
    NVFP4_UE8M0_SCALES = 8u,
    /* The w13 GEMM form.  By default the library chooses: from 512 routed
     * rows per expert on average (T*k >= 512*E), the tiles are computed by
     * pairs of CTAs (thread-block clusters of two sharing each tensor-core
     * MMA, M = 256: each CTA loads its own 128 activation rows and half of
     * the weight tile), with every expert's rows padded to 256; below that,
     * by single CTAs with rows padded to 128.  These flags force one form
     * (both together: NVFP4_ERR_INVALID_ARG).  The result is the same up to
     * the order of the FP32 accumulation inside the tensor cores. */
    NVFP4_W13_ONE_SM = 16u,
    NVFP4_W13_TWO_SM = 32u,
};

/* One-line description of the last error raised on the calling thread. */
const char *nvfp4_last_error_string(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int nvfp4_version(void);

/*
 * nvfp4_validate_scales -- the completeness check [page, ROOT CAUSE].
 *
 * A slot i of scales[n] (device, FP32, dequantisation direction) is bad if
 * written (device, one byte per slot, nullable) holds 0 at i, or the value is
 * NaN, +-inf, <= 0 or subnormal, or its FP32 reciprocal is not a finite normal
 * number.  ws: 256 bytes of device memory (256-byte aligned) for the
 * device-side result.  SYNCHRONOUS: waits for `stream`.  Results go to host
 * memory: *bad_count_host = number of bad slots, *first_bad_host = lowest bad
 * index or -1.  Returns NVFP4_OK when the check ran (whatever it found),
 * NVFP4_ERR_INVALID_ARG for n < 0, a null ws or null result pointers.
 */
int nvfp4_validate_scales(const float *scales, const uint8_t *written, int n, void *ws, nvfp4_stream_t stream,
                          int *bad_count_host, int *first_bad_host);

/*
 * nvfp4_quantize_experts -- dynamic activation quantisation of the routed
 * rows [page, §NVFP4 runtime-order figure; MoE section: SFScale[expert_idx]].
 *
 * x [T, H] BF16; topk_ids [T, k] int32 in [0, E); input_scale [E] FP32.
 * Routed row f = t*k + j goes to permuted row p (expert-major, ascending f
 * inside an expert) and is quantised with g = fl(1 / input_scale[e]):
 * per 16-block, s = e4m3(fl(fl(g*amax)/6)), q = e2m1(fl(fl(x*g)/s)), with
 * round-to-nearest-even and saturation; an all-zero-scale block gets code 0.
 * Outputs: q_out [R, H/2] packed codes; sf_out scales in `sf_layout`
 * (LINEAR: [R, H/16]; SWIZZLED: ceil(R/128) * ceil(H/64) * 512 bytes),
 * E4M3 bytes, or UE8M0 bytes when NVFP4_SF_UE8M0 is OR'ed into sf_layout;
 * expert_offsets [E+1] (first permuted row of each expert, [E] = R);
 * perm [R] (permuted row -> f).
 * SYNCHRONOUS: input_scale is validated first and the call waits for the
 * check; a bad slot returns NVFP4_ERR_SCALE_INVALID with no output written.
 * The call also waits for the quantiser and returns NVFP4_ERR_INVALID_ARG,
 * with no output written, if an expert id is outside [0, E).  Pointer
 * alignment: x 16 B, q_out 16 B, sf_out 4 B.  T*k*H/16 (the scale bytes)
 * must stay below 2^32 (else NVFP4_ERR_UNSUPPORTED_SHAPE).  Workspace:
 * nvfp4_quantize_workspace_size(T, k, E) bytes of device memory, 256-byte
 * aligned.
 */
size_t nvfp4_quantize_workspace_size(int T, int k, int E);
int nvfp4_quantize_experts(const uint16_t *x, int T, int H, const int32_t *topk_ids, int k, int E,
                           const float *input_scale, uint8_t *q_out, uint8_t *sf_out, int sf_layout,
                           int32_t *expert_offsets, int32_t *perm, void *ws, size_t ws_bytes,
                           nvfp4_stream_t stream);

/*
 * nvfp4_quantize_experts_static_scratch -- nvfp4_quantize_experts for callers
 * that cannot allocate device memory: a serving process whose memory pool has
 * already claimed the device (a cudaMalloc would fail or fragment it), or a
 * latency-critical path that must not call cudaMalloc / cudaFree because they
 * can synchronise the device.  The page has no counterpart; this is an
 * interface convenience of this library.
 *
 * Same arguments, outputs, checks and SYNCHRONOUS behaviour as
 * nvfp4_quantize_experts, minus the workspace: the scratch is one static
 * 4 MiB device array per GPU that loads the library, held until the process
 * exits.  That covers nvfp4_quantize_workspace_size(T, k, E) <= 4 MiB (about
 * 500,000 routed rows T*k with 128 experts); larger calls return
 * NVFP4_ERR_WORKSPACE_TOO_SMALL and write nothing.  The library calls no
 * cudaMalloc, cudaFree or other allocating routine on this path.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.  The cached address belongs
 *     to the device's primary context: after cudaDeviceReset on a device that
 *     has called this entry point, the process must not call it again on that
 *     device (the library's module, and the array, would be reloaded at
 *     another address).
 *   - Shapes the workspace entry point refuses are refused here with the
 *     same status (NVFP4_ERR_UNSUPPORTED_SHAPE); only the size limit above
 *     is particular to this entry point.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents (each call resets what it needs).  Calls whose work
 *     overlaps on the GPU -- e.g. from two host threads or on two streams --
 *     race on it and must be serialised by the caller.
 */
int nvfp4_quantize_experts_static_scratch(const uint16_t *x, int T, int H, const int32_t *topk_ids, int k, int E,
                                          const float *input_scale, uint8_t *q_out, uint8_t *sf_out, int sf_layout,
                                          int32_t *expert_offsets, int32_t *perm, nvfp4_stream_t stream);

/*
 * Expert weights of one MoE layer, canonical (checkpoint) layout
 * [page, glossary "Static weight quantization": packed FP4 weight, E4M3
 * weight_scale, FP32 weight_scale_2; §矩阵融合 "Gated FFN": gate and up fused
 * along the output dimension into w13].  All device pointers, [out, in] rows:
 *   w13_q [E, 2I, H/2]   rows 0..I-1 = gate, rows I..2I-1 = up
 *   w13_sf [E, 2I, H/16] linear E4M3 scales
 *   w13_scale2 [E]       weight_scale_2 (FP32)
 *   w13_input_scale [E]  stored activation scale of the w13 input
 *   w2_q [E, H, I/2], w2_sf [E, H, I/16], w2_scale2 [E], w2_input_scale [E]
 *   w13_input_written, w2_input_written: nullable [E] bytes, 0 = slot never
 *     written by the loader (checked with the values themselves).
 */
typedef struct {
    int E, H, I;
    const uint8_t *w13_q;
    const uint8_t *w13_sf;
    const float *w13_scale2;
    const float *w13_input_scale;
    const uint8_t *w13_input_written;
    const uint8_t *w2_q;
    const uint8_t *w2_sf;
    const float *w2_scale2;
    const float *w2_input_scale;
    const uint8_t *w2_input_written;
} nvfp4_moe_weights;

/*
 * nvfp4_prepare_weights -- one-time layout conversion of the weight scales
 * [page, "Kernel Backend": after choosing a backend the packed weights and
 * scales are converted to the layout that kernel wants].  Writes the w13 and
 * w2 block scales into `prepared` (device, nvfp4_prepared_weights_size bytes,
 * 256-byte aligned) in the swizzled tensor-core layout: 128-row x 64-K
 * tiles; for w13, the gate block and the up block of each 128 h columns
 * interleaved per 64-K step (a final 64 gate + 64 up block when I is an odd
 * multiple of 64).
 * The packed codes are used in place from nvfp4_moe_weights.  Asynchronous.
 */
size_t nvfp4_prepared_weights_size(int E, int H, int I);
int nvfp4_prepare_weights(const nvfp4_moe_weights *w, void *prepared, size_t prepared_bytes,
                          nvfp4_stream_t stream);

/*
 * nvfp4_prepare_weights_format -- nvfp4_prepare_weights for weights whose
 * block scales are in `format`: NVFP4_SF_E4M3 (as nvfp4_prepare_weights) or
 * NVFP4_SF_UE8M0, whose bytes are converted to the E4M3 encoding the tensor
 * cores take, relative to the largest scale of each weight row, with each
 * row's power of two stored after the scale tiles (see NVFP4_UE8M0_SCALES;
 * nvfp4_prepared_weights_size includes that room for either format).  The
 * last 256 bytes of `prepared` record
 * the format; nvfp4_moe_forward checks it against its flags.  Any other
 * format: NVFP4_ERR_INVALID_ARG.  Asynchronous.
 */
int nvfp4_prepare_weights_format(const nvfp4_moe_weights *w, void *prepared, size_t prepared_bytes, int format,
                                 nvfp4_stream_t stream);

/*
 * nvfp4_moe_forward -- the expert path of one MoE layer.
 *
 * x [T, H] BF16, topk_ids [T, k] int32, topk_weights [T, k] FP32 (device).
 * out [T, H] FP32 (device):
 *   out[t] = sum_j topk_weights[t, j] * W2_e(q2(silu(gate_e) * up_e))
 * with gate_e, up_e = W13_e(q1(x[t])), e = topk_ids[t, j], q1/q2 the NVFP4
 * activation quantisation with a1_gscale = 1/w13_input_scale[e] and
 * a2_gscale = 1/w2_input_scale[e], and every GEMM a block-scaled FP4 x FP4
 * product accumulated in FP32 and scaled by 1/(a_gscale * w_gscale).
 * Before any reciprocal is taken the 4E scale slots (w13/w2 input scales and
 * weight_scale_2) are validated; unless NVFP4_SCALES_PREVALIDATED is set the
 * call SYNCHRONISES on that check and returns NVFP4_ERR_SCALE_INVALID with
 * nothing launched after it and `out` untouched.
 * `prepared` is the output of nvfp4_prepare_weights for the same weights.
 * An expert id outside [0, E) stops the call on the device before anything
 * is written to `out` (reported by nvfp4_moe_status / NVFP4_SYNC_CHECK as
 * NVFP4_ERR_INVALID_ARG).  Alignment: x and out 16 B, ws and prepared 256 B,
 * weight codes 16 B.  Workspace: nvfp4_moe_workspace_size(T, H, I, E, k)
 * bytes of device memory, 256-byte aligned; its contents after the call are
 * internal.  T == 0 is valid (nothing is written).
 * Ordering: the call's kernels read x, topk_ids, topk_weights, the weights
 * and `prepared` once the work queued before them on `stream` has completed
 * (small batches read them before the scale check's result is known, and
 * write only after it); those buffers must not change until the call's work
 * on `stream` has completed.
 */
size_t nvfp4_moe_workspace_size(int T, int H, int I, int E, int k);
int nvfp4_moe_forward(const nvfp4_moe_weights *w, const void *prepared, const uint16_t *x, int T,
                      const int32_t *topk_ids, const float *topk_weights, int k, float *out, void *ws,
                      size_t ws_bytes, unsigned flags, nvfp4_stream_t stream);

/*
 * nvfp4_moe_forward_profiled -- nvfp4_moe_forward that also records six
 * caller-created CUDA events (events[i] is a cudaEvent_t) on `stream`:
 * [0] before the scale check, [1] after it, [2] after the token reorder,
 * [3] after the a1 quantiser, [4] after the w13 GEMM, [5] after the w2 GEMM,
 * so that each stage's device time is the gap between consecutive events.
 * A call that returns early records only the events before its exit point.
 */
int nvfp4_moe_forward_profiled(const nvfp4_moe_weights *w, const void *prepared, const uint16_t *x, int T,
                               const int32_t *topk_ids, const float *topk_weights, int k, float *out, void *ws,
                               size_t ws_bytes, unsigned flags, nvfp4_stream_t stream, void *const *events);

/*
 * nvfp4_moe_forward_host -- the same layer with HOST activations and routing:
 * copies x_host [T, H] BF16, topk_ids_host [T, k], topk_weights_host [T, k]
 * into the workspace, runs the layer and copies out [T, H] FP32 back to
 * out_host.  From 4096 tokens on, the tokens are processed in up to 8 chunks
 * (2048 first and last, up to 4096 between), each chunk's copy-in and the
 * previous chunk's copy-out overlapping the layer on other streams (tokens
 * are independent, so the result is that of one call).  Host buffers should
 * be page-locked for the copies to overlap.  SYNCHRONOUS: returns after
 * out_host is written and no copy of the call is in flight, also on error.
 * The scale check follows `flags` for the first chunk and runs on the device
 * for every chunk; a failure in any chunk is returned (its part of out_host
 * is then unspecified).  Not reentrant per device: concurrent calls on one
 * device serialise.  Workspace: nvfp4_moe_host_workspace_size(T, H, I, E, k)
 * bytes.
 */
size_t nvfp4_moe_host_workspace_size(int T, int H, int I, int E, int k);
int nvfp4_moe_forward_host(const nvfp4_moe_weights *w, const void *prepared, const uint16_t *x_host,
                           int T, const int32_t *topk_ids_host, const float *topk_weights_host, int k,
                           float *out_host, void *ws, size_t ws_bytes, unsigned flags,
                           nvfp4_stream_t stream);

/*
 * nvfp4_moe_status -- SYNCHRONOUS: waits for `stream`, then reports the
 * device-side status of the last nvfp4_moe_forward that used `ws`:
 * NVFP4_OK, NVFP4_ERR_SCALE_INVALID (bad slot found on the device; then
 * *first_bad_host is its index in the order w13_input_scale[E],
 * w2_input_scale[E], w13_scale2[E], w2_scale2[E]), NVFP4_ERR_INVALID_ARG
 * (an expert id outside [0, E)) or NVFP4_ERR_DEVICE_TIMEOUT.
 * first_bad_host is nullable.
 */
int nvfp4_moe_status(const void *ws, nvfp4_stream_t stream, int *first_bad_host);

/*
 * Intermediates of the last nvfp4_moe_forward on `ws`, for inspection
 * (device pointers into ws; valid until the next call on ws):
 *   a1q [rows_cap, H/2], sf1 (swizzled, ceil(H/64) tiles per 128 rows),
 *   a2q [rows_cap, I/2], sf2 (swizzled, 4*ceil(I/256) tiles per 128 rows),
 *   row_of [R] (routed row f -> padded permuted row), offsets [E+1] (compact),
 *   pad_offsets [E+1] (padded: every expert starts on a 128-row boundary,
 *   or a 256-row boundary when the w13 GEMM ran on CTA pairs),
 *   h [rows_cap, I] FP32, the SiLU(gate)*up intermediate (written only when
 *   a forward ran with NVFP4_DEBUG_KEEP_H, which needs
 *   nvfp4_moe_host_workspace_size(...) + rows_cap*I*4 bytes of workspace).
 * Returns NVFP4_ERR_INVALID_ARG if ws is null.
 */
enum { NVFP4_DEBUG_KEEP_H = 4u };
typedef struct {
    int rows_cap;
    uint8_t *a1q, *sf1, *a2q, *sf2;
    int32_t *row_of, *offsets, *pad_offsets;
    float *h;
} nvfp4_moe_intermediates;
int nvfp4_moe_intermediates_of(void *ws, int T, int H, int I, int E, int k,
                               nvfp4_moe_intermediates *out_host);

/*
 * nvfp4_residual_rmsnorm -- between stacked layers (not on the page):
 * x_next = bf16(r / sqrt(mean(r^2) + eps)), r = x + out, gamma = 1, per token.
 * x [T, H] BF16, out [T, H] FP32, x_next [T, H] BF16 (may alias x).
 */
int nvfp4_residual_rmsnorm(const uint16_t *x, const float *out, int T, int H, float eps,
                           uint16_t *x_next, nvfp4_stream_t stream);

/*
 * W4A16 expert forward -- the same layer with the weights kept NVFP4 and the
 * activations BF16 [page "Gemma 4 NVFP4 MoE 空输出", backend figure: the
 * MARLIN path executes the NVFP4 checkpoint as W4A16 and consumes no
 * activation input_scale].  Per routed row (token t, expert e):
 *   gate, up = x[t] . W13[e]^T,  W = e2m1(code) * e4m3(block scale) * weight_scale_2
 *   h        = bf16( SiLU(gate) * up )      (the activations stay 16-bit)
 *   out[t]  += topk_weights[t, j] * (h . W2[e]^T)
 * BF16 x BF16 tensor-core products with FP32 accumulation; out [T, H] FP32.
 * w13_input_scale / w2_input_scale are not read (they may be null); the
 * weight_scale_2 slots are validated as in nvfp4_moe_forward.
 *
 * nvfp4_w4a16_prepared_size / nvfp4_prepare_weights_w4a16: the weights' block
 * scales rearranged for this path ([E * N / 64][K / 64][64 rows][4 bytes] per
 * projection); device memory, 256-byte aligned, owned by the caller, valid
 * while the weights are unchanged.  Asynchronous on `stream`.
 * nvfp4_moe_w4a16_workspace_size: device workspace of the forward (256-byte
 * aligned).  nvfp4_moe_forward_w4a16: arguments, flags, synchronisation and
 * errors as nvfp4_moe_forward (the same shape limits apply).
 * nvfp4_moe_w4a16_intermediates_of: pointers, inside a workspace, to the
 * gathered BF16 rows [rows_cap, H] and to h [rows_cap, I] (padded permuted
 * row order, as nvfp4_moe_intermediates_of describes).
 */
size_t nvfp4_w4a16_prepared_size(int E, int H, int I);
int nvfp4_prepare_weights_w4a16(const nvfp4_moe_weights *w, void *prepared, size_t prepared_bytes,
                                nvfp4_stream_t stream);
size_t nvfp4_moe_w4a16_workspace_size(int T, int H, int I, int E, int k);
int nvfp4_moe_forward_w4a16(const nvfp4_moe_weights *w, const void *prepared, const uint16_t *x, int T,
                            const int32_t *topk_ids, const float *topk_weights, int k, float *out, void *ws,
                            size_t ws_bytes, unsigned flags, nvfp4_stream_t stream);
int nvfp4_moe_w4a16_intermediates_of(void *ws, int T, int H, int I, int E, int k, uint16_t **a16,
                                     uint16_t **h16);

/*
 * nvfp4_router_topk -- the MoE router [page "Gemma 4 NVFP4 MoE 空输出",
 * §矩阵融合 "MoE FFN": the routing result picks each token's experts and the
 * expert outputs are summed with the routing weights; page
 * "genesis-vllm-patches" (mlqm.cn), §3.3 patch P31: softmax and top-k on
 * logits upcast to FP32].  Per token t:
 *   topk_ids[t, 0..k)     the k experts of largest softmax probability, largest
 *                         first; equal logits go to the lower expert index
 *   topk_weights[t, 0..k) their probabilities renormalised over the k (they sum
 *                         to 1), i.e. the softmax of the k selected logits, FP32
 * logits: device, [T, E] row-major, FP32 (logits_dtype NVFP4_LOGITS_F32) or
 * BF16 (NVFP4_LOGITS_BF16, widened exactly to FP32); finite values (NaN or inf
 * logits give unspecified results).  topk_ids [T, k] int32 and
 * topk_weights [T, k] FP32 are device buffers owned by the caller, in the
 * layout nvfp4_moe_forward() reads.  Limits: T >= 0, 1 <= E <= 1024,
 * 1 <= k <= min(32, E).  Needs no workspace; asynchronous on `stream`.
 * Returns NVFP4_OK (T = 0 launches nothing), NVFP4_ERR_INVALID_ARG (shape,
 * dtype, null or misaligned pointer), NVFP4_ERR_CUDA (launch failure).
 */
int nvfp4_router_topk(const void *logits, int logits_dtype, int T, int E, int k, int32_t *topk_ids,
                      float *topk_weights, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_weights -- static weight quantisation on the device
 * [page, glossary "Static weight quantization"]: for each of `count` tensors
 * w [count, N, K] BF16 (K % 16 == 0), weight_scale_2[c] = fl(amax_c / 2688)
 * (2688 = 6 * 448, [page, §NVFP4 two-level scale]), then every row is block
 * quantised with g = fl(1 / weight_scale_2[c]) exactly as activations are.
 * Outputs q [count, N, K/2], sf [count, N, K/16] (linear), scale2 [count].
 * Workspace: nvfp4_quantize_weights_workspace_size(count) bytes.
 */
size_t nvfp4_quantize_weights_workspace_size(int count);
int nvfp4_quantize_weights(const uint16_t *w, int count, int N, int K, uint8_t *q, uint8_t *sf,
                           float *scale2, void *ws, size_t ws_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_weights_format -- nvfp4_quantize_weights with the block-scale
 * format chosen: sf_format 0 writes E4M3 scales (as nvfp4_quantize_weights),
 * NVFP4_SF_UE8M0 writes UE8M0 scales (see NVFP4_SF_UE8M0; weight_scale_2 and
 * the codes' rule are unchanged).  Any other sf_format: NVFP4_ERR_INVALID_ARG.
 */
int nvfp4_quantize_weights_format(const uint16_t *w, int count, int N, int K, int sf_format, uint8_t *q,
                                  uint8_t *sf, float *scale2, void *ws, size_t ws_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_selftest_block_division -- host-side exhaustive check of the exact
 * block-scale division used by the quantisers: for every finite non-zero
 * E4M3 scale s and every FP32 significand y in [1, 2), the two-constant
 * product fma(y, zh(s), y*zl(s)) must equal the correctly rounded y / s
 * (N. Brisebarre, J.-M. Muller, S. K. Raina, "Accelerating correctly rounded
 * floating-point division when the divisor is known in advance", IEEE Trans.
 * Computers 53(8), 2004).  Returns the number of mismatches (0 = exact);
 * nthreads <= 0 uses every host core.  Runs on the CPU only.
 */
long long nvfp4_selftest_block_division(int nthreads);

/*
 * nvfp4_selftest_ue8m0_carry -- the per-row carry of UE8M0 scales to the
 * tensor cores (NVFP4_UE8M0_SCALES), for every byte b and row shift c in
 * 0 .. 255: out (device, 131072 bytes, 4-byte aligned) receives
 * out[c * 256 + b] from the one-byte routine the weight preparation uses and
 * out[65536 + c * 256 + b] from the four-byte routine the GEMM uses.  The
 * carried byte is the E4M3 encoding of 2^(b - c - 7) when 1 <= b - c <= 15,
 * and 0 when b <= c.  Synchronous.  NVFP4_ERR_INVALID_ARG for a null or
 * misaligned `out`.
 */
int nvfp4_selftest_ue8m0_carry(uint8_t *out, nvfp4_stream_t stream);

/*
 * nvfp4_selftest_device_wait -- the failure path of the device-side waits,
 * run on purpose.  One small kernel waits on a barrier that nothing arrives
 * on: one thread gives up after limit_us microseconds (1 .. 10^6), a second,
 * with a ten times longer limit, gives up as soon as the first raises the
 * CTA's abort flag.  They record the expiry in the status block at the start
 * of `ws` (device, 256-byte aligned, at least 256 bytes) as the GEMM kernels
 * do, so nvfp4_moe_status(ws) then returns NVFP4_ERR_DEVICE_TIMEOUT and the
 * context stays usable.  Asynchronous; NVFP4_ERR_INVALID_ARG for a bad ws or
 * limit.
 */
int nvfp4_selftest_device_wait(void *ws, size_t ws_bytes, unsigned limit_us, nvfp4_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_MOE_H */
