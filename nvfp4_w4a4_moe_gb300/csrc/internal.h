// Host-side declarations shared by the translation units of libnvfp4moe.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace nvfp4 {

// ---------------------------------------------------------------- workspace
// Every region starts on a 256-byte boundary.
struct WsLayout {
    int T, H, I, E, k, R;
    int rows_cap, mtiles_cap, nchunks;
    int kc1, kc2;  // 64-element scale chunks per 128-row tile for a1 (H) and a2 (I)
    size_t hdr, g1, g2, alpha1, alpha2, counts, offsets, pad_off, chunk_hist, row_of, perm, row_src,
        tile_expert, live_mtiles, row_max, a1q, sf1, a2q, sf2, end;
    // forward_host staging (after `end`), and the optional FP32 h dump
    size_t x_stage, ids_stage, w_stage, out_stage, status_stage, host_end;
};

constexpr int kMaxHostChunks = 8;  // token chunks of the pipelined host entry point

constexpr int kRouteChunk = 2048;  // routed rows per routing CTA

// The w13 GEMM runs on CTA pairs (rows padded to 256 per expert) from this many
// routed rows per expert on average; below it, on single CTAs.  Measured on the
// 128-expert layer: pairs take 156 us against 160 at 8192 tokens (512 rows per
// expert), but 107 against 100 at 4096 and 84 against 71 at 2048, where the
// padding to 256 rows costs more than the pairs save.
constexpr long long kPairRowsPerExpert = 512;

// Up to this many routed rows (T*k), the w13 GEMM takes its small-batch plan:
// 64-column tiles, the A stage holding an m-tile's first 32 rows (no m-tile
// can hold more), and a deeper ring.
constexpr long long kSmallPlanRows = 32;
// Up to this many routed rows the w2 GEMM takes its small-batch plan: A in
// the ring (an m-tile's first 64 rows), a deeper ring, the combine from
// registers.
constexpr long long kSmallPlanRowsW2 = 64;
// The w13 small-batch plan quantises its A rows itself (no a1 quantiser
// launch) when every CTA gets one tile and K is at most this: the m-tile's
// 32 rows of all K slices stay in shared memory for the whole kernel.
constexpr long long kInlineQuantMaxK = 3072;
// Up to this many routed rows (and E <= 1024) the w13 GEMM on single CTAs
// routes its own tiles and starts its weight loads before its dependency wait.
constexpr long long kEarlyRows = 128;

WsLayout make_layout(int T, int H, int I, int E, int k);

// ---------------------------------------------------------------- kernels
struct ValidateArgs {
    const float *s[4];
    const uint8_t *written[4];
    float *recip[4];  // FP32 reciprocal of each slot (nullable per array)
    int E, narrays;
    float *alpha1, *alpha2;  // 1/(g_a * g_w) per expert (forward only; nullable)
    const uint32_t *prep_tag;  // format word of the prepared weights (nullable)
    uint32_t prep_tag_want;    // the value it must hold, else status 4
    DevHeader *hdr;
};
cudaError_t launch_validate(const ValidateArgs &a, cudaStream_t st);

struct RouteArgs {
    const int32_t *ids;
    int R, k, E, nchunks;
    int *chunk_hist, *counts, *offsets, *pad_off, *tile_expert;
    int *row_of;       // f -> output row (padded rows when `padded`, else compact)
    int *perm;         // compact permuted row -> f (nullable)
    int *row_src;      // padded row -> f, -1 for padding (nullable)
    int *offsets_out;  // caller copy of the compact offsets (nullable)
    int *row_max;      // UE8M0 forward: two arrays of rows_cap ints set to 0 for every padded row (nullable)
    int rows_cap;
    int pad_rows;      // expert row padding: 128, or 256 for the 2-SM w13 GEMM (m-tile pairs of one expert)
    int *live_mtiles;  // the 128-row m-tiles that hold rows, in order (nullable); count in hdr->num_live_mtiles
    int padded;
    DevHeader *hdr;
    // one-CTA routing: let the next kernel be scheduled only after this one's
    // dependency wait, so that it may read the call's inputs before its own
    // (the w13 GEMM that routes itself)
    int trigger_after_wait;
};
cudaError_t launch_route(const RouteArgs &a, cudaStream_t st);
// The scale check then the routing: one kernel when the routing takes one CTA
// (at most kRouteChunk routed rows), else the two launches above.
cudaError_t launch_validate_route(const ValidateArgs &v, const RouteArgs &a, cudaStream_t st);

struct QuantArgs {
    const uint16_t *x;
    const int32_t *ids;
    const int *row_of;
    const float *g;  // per-expert global scale
    int T, H, k;
    uint8_t *q;
    uint8_t *sf;
    int sf_swizzled, sf_kc;
    int sf_ue8m0;  // 0: E4M3 block scales; 1: UE8M0 bytes
    int *row_max;  // UE8M0: per padded row, the largest scale byte (atomicMax; nullable)
    DevHeader *hdr;  // read for the status; mode 2 writes a range error into it
    // forward, E4M3, at most kEarlyRows routed rows, rows padded to 128 per
    // expert: the kernel forms the row map (one m-tile per busy expert) and
    // the global scales (1/in_scale, as the scale check) from the call's
    // inputs and runs beside the routing kernel, whose completion it awaits
    // only before it exits; row_of and g are not read
    int self_route;
    const float *in_scale;
    int E;
};
cudaError_t launch_quant_experts(const QuantArgs &a, cudaStream_t st);

struct PrepArgs {
    const uint8_t *sf;  // canonical [E, N, K/16]
    uint8_t *out;       // [E][N/128 blocks][kc][512]; w13 blocks of one tile interleaved per K step
    int E, N, K, kc;
    int gate_up_I;      // w13: I > 0 (blocks of 128 gate rows and 128 up rows; a 64 + 64 tail block)
    int ue8m0;          // the canonical bytes are UE8M0: written carried per row (ue8m0_carried)
    float *row_factor;  // UE8M0: [E * N] per weight row 2^(shift - 117), written here, read by the epilogues
};
cudaError_t launch_prep_sf(const PrepArgs &a, cudaStream_t st);

cudaError_t launch_rmsnorm(const uint16_t *x, const float *out, int T, int H, float eps, uint16_t *xn,
                           cudaStream_t st);
// A kernel whose bounded waits run out by design (status 5 in hdr).
cudaError_t launch_wait_selftest(DevHeader *hdr, uint64_t limit_ns, cudaStream_t st);
// out [2][256 shifts][256 bytes]: the UE8M0 row carry of every byte and shift, by the
// one-byte and the four-byte routine.
cudaError_t launch_ue8m0_carry_selftest(uint8_t *out, cudaStream_t st);

// Router: softmax / top-k / renormalise over logits [T, E] (FP32, or BF16 when bf16 != 0).
cudaError_t launch_router_topk(const void *logits, int bf16, int T, int E, int k, int32_t *ids, float *w,
                               cudaStream_t st);

cudaError_t launch_quantize_weights(const uint16_t *w, int count, int N, int K, uint8_t *q, uint8_t *sf,
                                    float *scale2, unsigned *amax_bits, int ue8m0, cudaStream_t st);

struct GemmArgs {
    // A: activations [rows_cap, K/2]; B: weights [E * Nrows, K/2]
    const uint8_t *a_q, *b_q;
    const uint8_t *a_sf, *b_sf;  // swizzled scale tiles
    int rows_cap, K, N, E;
    int a_kc, b_kc;
    int gate_up_I;  // w13: I > 0 (B tile = up to 128 gate rows + the matching up rows)
    const int *tile_expert, *pad_off, *counts;
    const float *alpha;
    // w13 epilogue (SiLU * up, requantise)
    const float *g2;
    uint8_t *a2q, *sf2;
    int I, kc2;
    float *h_dump;
    int ue8m0;        // UE8M0 block scales: A carried per row, B prepared per row, factors in the epilogue
    const int *a_row_max;      // UE8M0: the A rows' largest scale bytes
    int *out_row_max;          // UE8M0, w13: the a2 rows' largest scale bytes (atomicMax; zero on entry)
    const float *b_row_factor; // UE8M0: [E * N] weight-row factors 2^(shift - 117)
    float *zero_out;  // w13 kernel: [T, H] FP32 output cleared for the w2 kernel's reductions (nullable)
    long long zero_floats;
    // w2 epilogue (weighted combine)
    const int *row_src;
    const float *topk_w;
    int k, H;
    float *out;
    DevHeader *hdr;
    int mtiles_cap;
    int pairs;                 // w13: CTA pairs on m-tile pairs (rows padded to 256 per expert)
    int small;                 // the small-batch plan (w13: at most kSmallPlanRows routed rows, w2: kSmallPlanRowsW2)
    // w13 small-batch plan, a_inline: the kernel routes its own tile from the
    // call's inputs (ids, the input and weight scales), quantises A from x
    // (also writing it to a_q / a_sf), and runs its loads and MMAs before its
    // dependency wait; only its writes wait for the scale check and routing
    int a_inline;
    const uint16_t *x;         // BF16 tokens [T, K]
    const int32_t *ids;        // top-k ids [R]
    int R;
    const float *in_scale1, *in_scale2, *w13_scale2;  // w13_input_scale, w2_input_scale, w13 weight_scale_2 [E]
    // w13 on single CTAs, E4M3, at most kEarlyRows routed rows (E <= 1024):
    // the kernel routes its tiles from the ids (one m-tile per busy expert)
    // and issues the weight loads of its first ring stages before its
    // dependency wait; their A loads and everything else follow the wait
    int early;
    const int *live_mtiles;    // w2: the m-tiles holding rows, in order (nullable: all m-tiles)
};
cudaError_t launch_gemm_w13(const GemmArgs &a, cudaStream_t st);
cudaError_t launch_gemm_w2(const GemmArgs &a, cudaStream_t st);

// W4A16 expert GEMMs: BF16 activation rows against NVFP4 weights.
struct W16Args {
    const uint16_t *a;       // A: BF16 rows [rows_cap, K]
    const uint8_t *b_q;      // B: FP4 codes [E * N, K/2]
    const uint8_t *b_sfp;    // B scales, prepared: [E][N/64][K/64][64 rows][4 bytes]
    int rows_cap, K, N, E;
    int gate_up_I;           // w13: I (B tile = up to 128 gate rows + the matching up rows); w2: 0
    const int *tile_expert, *pad_off, *counts, *row_src;
    const float *scale2;     // weight_scale_2 per expert: the epilogue's multiplier
    uint16_t *h;             // w13: h [rows_cap, I] BF16
    int I;
    const float *topk_w;     // w2: combine
    int k, H;
    float *out;
    DevHeader *hdr;
    int mtiles_cap;
    int col_group;           // w2: output column blocks per tile group (divides N / 128)
};
cudaError_t launch_w16_w13(const W16Args &a, cudaStream_t st);
cudaError_t launch_w16_w2(const W16Args &a, cudaStream_t st);
// A rows of the W4A16 path: padded permuted row p holds x[row_src[p] / k] (zero on padding rows);
// also clears out [out_floats] (a multiple of 4) when the device status is clean.
cudaError_t launch_gather_rows(const uint16_t *x, int H, int k, const int *row_src, const DevHeader *hdr,
                               int rows_cap, uint16_t *a, float *out, long long out_floats, cudaStream_t st);
// W4A16 weight-scale layout: canonical [E, N, K/16] -> [E][N/64][K/64][64][4].
cudaError_t launch_prep_sf_w16(const uint8_t *sf, uint8_t *out, int E, int N, int K, cudaStream_t st);

// 2-D byte tensor map [rows, row_bytes], box (box_bytes x box_rows), 128-byte swizzle or none.
bool make_tensor_map_2d(CUtensorMap *m, const void *base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
                        uint32_t box_rows, bool swizzle128);

// ---------------------------------------------------------------- helpers
// Launch with programmatic stream serialisation (see pdl_wait / pdl_trigger).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// The shape checks of nvfp4_quantize_experts (status and error text as that
// entry point returns them): NVFP4_OK or NVFP4_ERR_UNSUPPORTED_SHAPE.
int quantize_shape_status(int T, int H, int k, int E);

const DivTable &div_table();
int sm_count();
void set_error(const char *fmt, ...);

}  // namespace nvfp4
