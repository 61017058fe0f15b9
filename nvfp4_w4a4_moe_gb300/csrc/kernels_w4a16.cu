// W4A16 expert GEMMs: NVFP4 weights (E2M1 codes, E4M3 block scales, FP32
// weight_scale_2) against BF16 activations, on the tcgen05 tensor cores.
//
// Page cited: "Gemma 4 NVFP4 MoE 空输出" (taking-lying-flat.github.io):
//   backend overview: the MARLIN path runs NVFP4 checkpoints as W4A16, the
//   weights stay 4-bit and the activations 16-bit, and it consumes no
//   activation input_scale; §矩阵融合 "Gated FFN" / "MoE FFN": the same
//   gate/up GEMM, act(gate) * up, down GEMM and weighted combine as the W4A4
//   path.
//
// The weights stay FP4 in memory.  Each stage, converter warps expand the
// stage's FP4 weight tile into a BF16 tile in shared memory, in the 128-byte
// swizzled K-major layout the MMA reads: code value times E4M3 block scale
// has at most 6 significant bits, so the product is exact in BF16, and the
// FP32 weight_scale_2 is applied in the epilogue.  The MMA is
// tcgen05.mma.kind::f16 with BF16 A and B and FP32 accumulators; with no
// block scales in TMEM, two accumulators fit in both kernels.
//
// Kernel shape (one persistent CTA per SM):
//   warp 0     TMA producer: per 64-K stage the A tile (128 BF16 rows x 128 B,
//              128-byte swizzle), the FP4 codes of the B tile (64-row boxes of
//              32 B) and its scales (256-byte bulk copies of the prepared
//              layout), into a ring of 6 (w13) or 5 (w2) stages.
//   warp 1     TMEM owner and MMA issuer: 4 x kind::f16 K16 per stage, M128 x
//              N256 (w13: 128 gate + 128 up rows) or N128 (w2).
//   warps 2-17 converters: FP4 codes x block scale -> BF16 tile in a second,
//              two-slot ring (byte permutes on register-held tables, then
//              BF16 products), a proxy fence and an arrive on the slot's
//              "ready" barrier; the MMA frees both rings' slots by commits.
//   the rest   epilogue (4 warps for w13, 2 x 4 for w2): w13 forms
//              h = SiLU(s2 gate) (s2 up) and stores it as
//              BF16 (the second GEMM's A operand); w2 scatters
//              w * s2 * y2 into the token-order FP32 output with vector
//              reductions, as in the W4A4 path.
// Every wait is bounded (%globaltimer); on expiry the kernel records the
// error in the workspace header, drains what it has in flight and exits.
#include <climits>

#include "internal.h"
#include "tc_common.cuh"

// Warp counts: the conversion is latency-bound per warp (measured 1.88 ms
// per prefill call with 4 converter warps, 1.45 with 8, 1.31 with 16), so the
// converters take most of the CTA; with two accumulators one epilogue warp
// per TMEM lane quarter (w13) or two groups of four (w2) keep up.
#ifndef W16_CONV_WARPS
#define W16_CONV_WARPS 16
#endif
#ifndef W16_EPI13
#define W16_EPI13 4
#endif
#ifndef W16_EPI2
#define W16_EPI2 8
#endif

namespace nvfp4 {
namespace {

using namespace tc;

constexpr int WBM = 128, WBK = 64;         // K per stage: one 128-byte row of BF16
constexpr int W_A_BYTES = WBM * WBK * 2;   // 16 KB
constexpr int W_TMEM_COLS = 512;
constexpr int kConvWarps = W16_CONV_WARPS;
constexpr int kXposeLd = 33;
constexpr uint64_t kWLimitNs = 1000000000ull;
constexpr uint64_t kWDrainNs = 200000000ull;

// Two rings: NS stages of the TMA-loaded tiles (A, FP4 codes, scales; small,
// so the loads run well ahead) and NB stages of converted BF16 B tiles.
template <int EPI>
struct WPlan {
    static constexpr int BN = EPI == 0 ? 256 : 128;
    static constexpr int NS = EPI == 0 ? 6 : 5;
    static constexpr int NB = 2;
    static constexpr int NUM_EPI_WARPS = EPI == 0 ? W16_EPI13 : W16_EPI2;
    static constexpr int Q_PARTS = NUM_EPI_WARPS / (4 * (EPI == 0 ? 1 : 2));  // warps per TMEM lane quarter and group
    static constexpr int EPI_THREADS = 32 * NUM_EPI_WARPS;
    static constexpr int EPI_GROUPS = EPI == 0 ? 1 : 2;
    static constexpr int CONV_WARP0 = 2;
    static constexpr int EPI_WARP0 = CONV_WARP0 + kConvWarps;
    static constexpr int NUM_THREADS = 32 * EPI_WARP0 + EPI_THREADS;
    static constexpr int ACC_BUFS = 2;
    static constexpr int B16_BYTES = BN * WBK * 2;  // BF16 B tile: BN rows x 128 B
    static constexpr int BQ_BYTES = BN * WBK / 2;   // FP4 codes: BN rows x 32 B
    static constexpr int SQ_BYTES = BN * 4;         // E4M3 scales: BN rows x 4
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B16 = OFF_A + NS * W_A_BYTES;
    static constexpr int OFF_BQ = OFF_B16 + NB * B16_BYTES;
    static constexpr int OFF_SQ = OFF_BQ + NS * BQ_BYTES;
    static constexpr int OFF_LUT = OFF_SQ + NS * SQ_BYTES;  // 128 x u32: E4M3 scale -> BF16x2
    static constexpr int OFF_BAR = OFF_LUT + 128 * 4;
    static constexpr int NUM_BARS = 2 * NS + 2 * NB + 2 * ACC_BUFS + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_XPOSE = (OFF_MISC + 16 + 15) & ~15;
    static constexpr int XPOSE_BYTES = EPI == 1 ? NUM_EPI_WARPS * 32 * kXposeLd * 4 : 0;
    static constexpr int SMEM_BYTES = OFF_XPOSE + XPOSE_BYTES + 1024;  // + alignment slack
    static_assert(ACC_BUFS * BN <= W_TMEM_COLS, "accumulators exceed TMEM");
    static_assert(W_A_BYTES % 1024 == 0 && B16_BYTES % 1024 == 0, "swizzled tiles keep 1024-byte alignment");
    static_assert(SMEM_BYTES <= 232448, "shared memory plan exceeds the opt-in limit");
};

// Instruction descriptor, kind::f16: FP32 accumulator (bits 4-5 = 1), BF16 A
// and B (code 1 at bits 7-9 and 10-12), K-major both, N>>3 at 17-22, M>>4 at
// 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(WBM >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Two BF16 products, each exact here (at most 6 significant bits).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Two FP32 values rounded to nearest-even BF16, packed (first in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float silu_w16(float z) { return __fdividef(z, 1.0f + __expf(fminf(-z, 80.0f))); }

// Tile geometry.  w13: tile t covers h columns [128 nt, 128 nt + hc), hc =
// min(128, I - 128 nt), B rows = hc gate rows then hc up rows, m-tile major.
// w2: output columns [128 nt, 128 nt + 128), in groups of col_group column
// blocks: within a group the m-tiles are walked with the group's column
// blocks adjacent.  A group's slice of the FP32 output stays in L2 for the
// combine's reductions, and each BF16 A tile is read once per group rather
// than once per column block.
struct WTile {
    int mt, nt, e, hc;
};
template <int EPI>
__device__ __forceinline__ WTile w_tile(const W16Args &p, int tile, int NT, int MT)
{
    WTile t;
    if (EPI == 0) {
        t.mt = tile / NT;
        t.nt = tile - t.mt * NT;
        t.hc = min(128, p.gate_up_I - 128 * t.nt);
    } else {
        const int G = p.col_group;
        const int grp = tile / (MT * G), rem = tile - grp * (MT * G);
        t.mt = rem / G;
        t.nt = grp * G + (rem - t.mt * G);
        t.hc = 128;
    }
    t.e = p.tile_expert[t.mt];
    return t;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Four E2M1 codes (the low 16 bits of c, code i in nibble i) -> their BF16
// values as two BF16x2 words (codes 0, 1 in o0; 2, 3 in o1), in registers.
// The page's table has magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, i.e. BF16 bits
// 0000 3F00 3F80 3FC0 4000 4040 4080 40C0; the low and high bytes of those
// eight values are held in two 8-byte tables, and byte permutes index them
// with each code's three magnitude bits.  The sign (code bit 3) is the top
// bit of a byte of c or of c << 4, which a sign-replicating permute spreads
// to the high bytes.
__device__ __forceinline__ void e2m1x4_bf16(uint32_t c, uint32_t &o0, uint32_t &o1)
{
    const uint32_t sel = c & 0x7777u;
    const uint32_t lo = prmt(0xC0800000u, 0xC0804000u, sel);
    const uint32_t hi = prmt(0x3F3F3F00u, 0x40404040u, sel) | (prmt(c << 4, c, 0xD9C8u) & 0x80808080u);
    o0 = prmt(lo, hi, 0x5140u);
    o1 = prmt(lo, hi, 0x7362u);
}
// BF16 bits of a non-negative E4M3 scale byte (exact: at most 4 significant bits).
__device__ __forceinline__ uint32_t e4m3_bf16(uint32_t b)
{
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    if (e == 15u && m == 7u) return 0x7FC0u;  // NaN
    const float v = e == 0u ? (float)m * 0x1p-9f : ldexpf((float)(8u + m), (int)e - 10);
    return __float_as_uint(v) >> 16;
}

template <int EPI>
__global__ void __launch_bounds__(WPlan<EPI>::NUM_THREADS, 1)
    w16_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const W16Args p)
{
    using P = WPlan<EPI>;
    constexpr int NS = P::NS, NB = P::NB, ACC_BUFS = P::ACC_BUFS, BN = P::BN, EPI_GROUPS = P::EPI_GROUPS,
                  EPI_THREADS = P::EPI_THREADS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P::OFF_BAR);
    // full / empty: the TMA ring; ready / bfree: the BF16 ring
    uint64_t *full = bars, *empty = bars + NS, *ready = bars + 2 * NS, *bfree = ready + NB, *acc_full = bfree + NB,
             *acc_empty = acc_full + ACC_BUFS, *drain = acc_empty + ACC_BUFS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + P::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + P::OFF_MISC + 4);
    uint32_t *lut_scale = reinterpret_cast<uint32_t *>(smem + P::OFF_LUT);  // E4M3 byte -> (s, s) as BF16x2

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Set-up that reads nothing the previous kernel writes runs before the
    // dependency wait, overlapping that kernel's tail.
    pdl_trigger();
    for (int i = threadIdx.x; i < 128; i += blockDim.x) {
        const uint32_t s = e4m3_bf16((uint32_t)i);
        lut_scale[i] = s | (s << 16);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < NB; ++s) {
            mbar_init(&ready[s], kConvWarps);
            mbar_init(&bfree[s], 1);
        }
        for (int i = 0; i < ACC_BUFS; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], EPI_THREADS / EPI_GROUPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(W_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    pdl_wait();  // the previous kernel's outputs (A operand, row maps, status)
    const int NT = EPI == 0 ? (p.gate_up_I + 127) / 128 : p.N / 128;
    const int MT = p.hdr->num_mtiles;
    const int ntiles = MT * NT;
    if (p.hdr->status != 0 || (int)blockIdx.x >= ntiles) {
        // nothing to do (same decision in every thread): give TMEM back
        if (warp == 1)
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(*tmem_slot), "r"(W_TMEM_COLS)
                         : "memory");
        return;
    }
    const int KT = p.K / WBK;
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t stage = 0, phase = 0, issued = 0, last_parity = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            const WTile ti = w_tile<EPI>(p, tile, NT, MT);
            const int rows_b = EPI == 0 ? 2 * ti.hc : 128;
            const uint32_t bytes = (uint32_t)W_A_BYTES + (uint32_t)rows_b * 36u;  // + 32 B codes, 4 B scales per row
            // first B row of each 64-row box: w13 gate rows then the matching up rows
            int brow[4];
            int nbox = 0;
            if (EPI == 0) {
                const int gate = ti.e * 2 * p.gate_up_I + 128 * ti.nt;
                for (int r = 0; r < ti.hc; r += 64) brow[nbox++] = gate + r;
                for (int r = 0; r < ti.hc; r += 64) brow[nbox++] = gate + p.gate_up_I + r;
            } else {
                brow[nbox++] = ti.e * p.N + 128 * ti.nt;
                brow[nbox++] = ti.e * p.N + 128 * ti.nt + 64;
            }
            for (int kt = 0; kt < KT; ++kt) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, kWLimitNs)) {
                    ok = false;
                    break;
                }
                uint64_t *fb = &full[stage];
                mbar_expect_tx(fb, bytes);
                tma_2d(smem + P::OFF_A + stage * W_A_BYTES, &tmap_a, kt * (WBK * 2), ti.mt * WBM, fb);
                uint8_t *bq = smem + P::OFF_BQ + stage * P::BQ_BYTES;
                uint8_t *sq = smem + P::OFF_SQ + stage * P::SQ_BYTES;
                for (int b = 0; b < nbox; ++b) {
                    tma_2d(bq + b * 64 * (WBK / 2), &tmap_b, kt * (WBK / 2), brow[b], fb);
                    bulk_g2s(sq + b * 64 * 4, p.b_sfp + ((size_t)(brow[b] / 64) * KT + kt) * 256, 256u, fb);
                }
                issued |= 1u << stage;
                last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            atomicOr(&p.hdr->error_flags, kErrTimeoutProducer);
        }
        for (int s = 0; s < NS; ++s)
            if (issued & (1u << s)) mbar_wait(&full[s], (last_parity >> s) & 1u, nullptr, kWDrainNs);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        uint32_t ts = 0, bs = 0, bphase = 0, acc = 0, acc_phase = 0;
        bool ok = true;
        const uint64_t da0 = desc_sw128(su32(smem + P::OFF_A)), db0 = desc_sw128(su32(smem + P::OFF_B16));
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            const int nt = tile % NT;
            const uint32_t idesc = idesc_f16(EPI == 0 ? 2 * min(128, p.gate_up_I - 128 * nt) : 128);
            if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag, kWLimitNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + acc * BN;
            for (int kt = 0; kt < KT; ++kt) {
                // the converters arrive on ready[bs] only after they have seen
                // the TMA stage land and written its BF16 B tile
                if (!mbar_wait(&ready[bs], bphase, abort_flag, kWLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t da = da0 + (uint64_t)(ts * (W_A_BYTES >> 4));
                const uint64_t db = db0 + (uint64_t)(bs * (P::B16_BYTES >> 4));
#pragma unroll
                for (int j = 0; j < 4; ++j) tc_mma_f16(d, da + 2 * j, db + 2 * j, idesc, (kt | j) != 0);
                tc_commit(&empty[ts]);  // A tile read (the converters finished with the codes before ready)
                tc_commit(&bfree[bs]);  // BF16 B tile read
                if (++ts == NS) ts = 0;
                if (++bs == NB) {
                    bs = 0;
                    bphase ^= 1u;
                }
            }
            if (!ok) break;
            tc_commit(&acc_full[acc]);
            if (++acc == ACC_BUFS) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (!ok) {
            *abort_flag = 1;
            atomicOr(&p.hdr->error_flags, kErrTimeoutMma);
        }
        tc_commit(drain);
        mbar_wait(drain, 0, nullptr, kWDrainNs);
    } else if (warp >= P::CONV_WARP0 && warp < P::EPI_WARP0) {
        // ------------------------------------------------ converters
        // 16-byte output chunk j of B row r holds K elements 8j..8j+7: codes
        // bytes 4j..4j+3 of the row, block scale j/2; it is stored at chunk
        // j ^ (r & 7) of the row, the 128-byte swizzle the descriptor names.
        // An item is one 16-element block: chunks 2jj and 2jj+1, scale jj.
        const int ct = threadIdx.x - 32 * P::CONV_WARP0;
        uint32_t ts = 0, tphase = 0, bs = 0, bphase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            const int nt = tile % NT;
            const int rows_b = EPI == 0 ? 2 * min(128, p.gate_up_I - 128 * nt) : 128;
            for (int kt = 0; kt < KT; ++kt) {
                if (!mbar_wait(&full[ts], tphase, abort_flag, kWLimitNs) ||
                    !mbar_wait(&bfree[bs], bphase ^ 1u, abort_flag, kWLimitNs)) {
                    ok = false;
                    break;
                }
                const uint32_t *bq = reinterpret_cast<const uint32_t *>(smem + P::OFF_BQ + ts * P::BQ_BYTES);
                const uint8_t *sq = smem + P::OFF_SQ + ts * P::SQ_BYTES;
                uint8_t *b16 = smem + P::OFF_B16 + bs * P::B16_BYTES;
                // one 16-element block (two 16-byte output chunks, one scale) per item
                const int items = rows_b * 4;
#pragma unroll 4
                for (int i = ct; i < items; i += 32 * kConvWarps) {
                    const int r = i >> 2, jj = i & 3;
                    const uint2 cw = reinterpret_cast<const uint2 *>(bq)[r * 4 + jj];
                    const uint32_t s2 = lut_scale[sq[r * 4 + jj] & 127u];
                    uint4 o0, o1;
                    e2m1x4_bf16(cw.x, o0.x, o0.y);
                    e2m1x4_bf16(cw.x >> 16, o0.z, o0.w);
                    e2m1x4_bf16(cw.y, o1.x, o1.y);
                    e2m1x4_bf16(cw.y >> 16, o1.z, o1.w);
                    o0.x = bf16x2_mul(o0.x, s2);
                    o0.y = bf16x2_mul(o0.y, s2);
                    o0.z = bf16x2_mul(o0.z, s2);
                    o0.w = bf16x2_mul(o0.w, s2);
                    o1.x = bf16x2_mul(o1.x, s2);
                    o1.y = bf16x2_mul(o1.y, s2);
                    o1.z = bf16x2_mul(o1.z, s2);
                    o1.w = bf16x2_mul(o1.w, s2);
                    uint8_t *row = b16 + r * 128;
                    *reinterpret_cast<uint4 *>(row + (((2 * jj) ^ (r & 7)) << 4)) = o0;
                    *reinterpret_cast<uint4 *>(row + (((2 * jj + 1) ^ (r & 7)) << 4)) = o1;
                }
                // generic-proxy stores -> visible to the tensor core's reads
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&ready[bs]);
                if (++ts == NS) {
                    ts = 0;
                    tphase ^= 1u;
                }
                if (++bs == NB) {
                    bs = 0;
                    bphase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(&p.hdr->error_flags, kErrTimeoutMma);
        }
    } else if (warp >= P::EPI_WARP0) {
        // ------------------------------------------------ epilogue
        const int ew = warp - P::EPI_WARP0;
        const int group = ew / (P::NUM_EPI_WARPS / EPI_GROUPS);
        const int quarter = warp & 3;   // TMEM lanes this warp may read
        const int part = (ew >> 2) % P::Q_PARTS;  // which slice of the tile's columns
        const int r_in = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        float *xp = reinterpret_cast<float *>(smem + P::OFF_XPOSE) + ew * 32 * kXposeLd;
        uint32_t acc = EPI_GROUPS == 2 ? (uint32_t)group : 0u, acc_phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x + group * gridDim.x; tile < ntiles; tile += EPI_GROUPS * gridDim.x) {
            const WTile ti = w_tile<EPI>(p, tile, NT, MT);
            const int e = ti.e;
            const int row = ti.mt * WBM + r_in;
            bool valid;
            float s0;  // w13: weight_scale_2; w2: routing weight * weight_scale_2
            int t = 0;
            if (EPI == 0) {
                valid = row < p.pad_off[e] + p.counts[e];
                s0 = p.scale2[e];
            } else {
                const int f = p.row_src[row];
                valid = f >= 0;
                s0 = valid ? __fmul_rn(p.topk_w[f], p.scale2[e]) : 0.0f;
                t = valid ? f / p.k : 0;
            }
            if (!mbar_wait(&acc_full[acc], acc_phase, abort_flag, kWLimitNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t col0 = lane_base + acc * BN;
            if (EPI == 0) {
                // h columns [w0, w0 + hw) of the tile, 32 at a time: gate at
                // accumulator column w0.., up at hc + w0..; the accumulator is
                // released once the last columns are in registers.
                const int hw = ti.hc / P::Q_PARTS, w0 = part * hw;
                for (int c = 0; 32 * c < hw; ++c) {
                    float gate[32], up[32];
                    tmem_ld16(col0 + w0 + 32 * c, gate);
                    tmem_ld16(col0 + w0 + 32 * c + 16, gate + 16);
                    tmem_ld16(col0 + ti.hc + w0 + 32 * c, up);
                    tmem_ld16(col0 + ti.hc + w0 + 32 * c + 16, up + 16);
                    tmem_wait_ld(gate, up);
                    if (32 * (c + 1) >= hw) {
                        tc_fence_before();
                        mbar_arrive(&acc_empty[acc]);
                    }
                    uint32_t hb[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float h0 = silu_w16(s0 * gate[2 * i]) * (s0 * up[2 * i]);
                        const float h1 = silu_w16(s0 * gate[2 * i + 1]) * (s0 * up[2 * i + 1]);
                        hb[i] = pack_bf16x2(h0, h1);
                    }
                    if (valid) {
                        uint4 *dst = reinterpret_cast<uint4 *>(p.h + (size_t)row * p.I + 128 * ti.nt + w0 + 32 * c);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(hb[4 * i], hb[4 * i + 1], hb[4 * i + 2], hb[4 * i + 3]);
                    }
                }
                if (++acc == ACC_BUFS) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            } else {
                // out[t, cols] += w * s2 * y2 on this warp's 64 columns, 32 at
                // a time, transposed through shared memory so each reduction
                // covers four contiguous 128-byte row segments
                const int sub = lane >> 3, cc = (lane & 7) * 4;
                constexpr int CW = 128 / P::Q_PARTS;  // columns of this warp
                for (int c2 = 0; c2 < CW / 32; ++c2) {
                    const int cbase = CW * part + 32 * c2;
                    float v[32];
                    tmem_ld16(col0 + cbase, v);
                    tmem_ld16(col0 + cbase + 16, v + 16);
                    tmem_wait_ld(v);
                    if (c2 == CW / 32 - 1) {
                        tc_fence_before();
                        mbar_arrive(&acc_empty[acc]);
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) xp[lane * kXposeLd + i] = v[i] * s0;
                    __syncwarp();
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int rr = it * 4 + sub;
                        const int t_r = __shfl_sync(0xffffffffu, t, rr);
                        const int ok_r = __shfl_sync(0xffffffffu, (int)valid, rr);
                        const float *src = xp + rr * kXposeLd + cc;
                        if (ok_r)
                            red_add_v4(p.out + (size_t)t_r * p.H + ti.nt * 128 + cbase + cc, src[0], src[1], src[2],
                                       src[3]);
                    }
                    __syncwarp();
                }
                acc_phase ^= 1u;  // each group owns one accumulator
            }
        }
        if (!ok) {
            *abort_flag = 1;
            atomicOr(&p.hdr->error_flags, kErrTimeoutEpilogue);
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(W_TMEM_COLS)
                     : "memory");
    }
}

// Padded permuted row p of the A operand = x[row_src[p] / k], zero on padding
// rows; one warp per row, 16 bytes per lane and step.  The FP32 output is
// cleared here for the w2 kernel's reductions, after the status check, so a
// refused call writes nothing.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t *__restrict__ x, int H, int k,
                                                          const int *__restrict__ row_src, const DevHeader *hdr,
                                                          uint16_t *__restrict__ a, float4 *__restrict__ out,
                                                          long long out4)
{
    pdl_trigger();
    pdl_wait();  // the routing kernel's row map and status
    if (hdr->status != 0) return;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < out4;
         i += (long long)gridDim.x * blockDim.x)
        out[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    const long long rows = (long long)hdr->num_mtiles * WBM;
    const int lane = threadIdx.x & 31;
    const int n16 = H / 8;  // 16-byte chunks per row
    for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows;
         r += ((long long)gridDim.x * blockDim.x) >> 5) {
        const int f = row_src[r];
        uint4 *dst = reinterpret_cast<uint4 *>(a + (size_t)r * H);
        if (f >= 0) {
            const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)(f / k) * H);
            for (int i = lane; i < n16; i += 32) dst[i] = __ldg(src + i);
        } else {
            for (int i = lane; i < n16; i += 32) dst[i] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// [E, N, K/16] scale bytes -> [E*N/64][K/64][64 rows][4 bytes]: the four
// scales of one 64-K step for 64 consecutive rows are one 256-byte run.
__global__ void __launch_bounds__(256) prep_sf_w16_kernel(const uint8_t *__restrict__ sf, uint8_t *__restrict__ out,
                                                          long long groups, int K)
{
    const int KT = K / 64, nsf = K / 16;
    const long long words = groups * KT * 64;
    for (long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x; w < words;
         w += (long long)gridDim.x * blockDim.x) {
        const long long g = w / ((long long)KT * 64);
        const int rem = (int)(w - g * KT * 64);
        const int kt = rem >> 6, rr = rem & 63;
        const long long row = g * 64 + rr;
        reinterpret_cast<uint32_t *>(out)[w] = *reinterpret_cast<const uint32_t *>(sf + row * nsf + 4 * kt);
    }
}

template <int EPI>
cudaError_t launch_w16(const W16Args &a, cudaStream_t st)
{
    // function attributes are per device: set once on each
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaError_t aerr = cudaGetDevice(&dev);
    if (aerr != cudaSuccess) return aerr;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        aerr = cudaFuncSetAttribute(w16_gemm_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    WPlan<EPI>::SMEM_BYTES);
        if (aerr != cudaSuccess) return aerr;
        attr_set[dev] = true;
    }
    CUtensorMap ma, mb;
    if (!make_tensor_map_2d(&ma, a.a, (uint64_t)a.K * 2, (uint64_t)a.rows_cap, 128, WBM, true))
        return cudaErrorInvalidValue;
    if (!make_tensor_map_2d(&mb, a.b_q, (uint64_t)a.K / 2, (uint64_t)a.E * (uint64_t)a.N, WBK / 2, 64, false))
        return cudaErrorInvalidValue;
    const long long nt = EPI == 0 ? (a.gate_up_I + 127) / 128 : a.N / 128;
    const long long tiles = (long long)a.mtiles_cap * nt;
    int grid = sm_count();
    if (tiles < grid) grid = (int)(tiles > 0 ? tiles : 1);
    const cudaError_t err = launch_pdl(w16_gemm_kernel<EPI>, dim3(grid), dim3(WPlan<EPI>::NUM_THREADS),
                                       WPlan<EPI>::SMEM_BYTES, st, ma, mb, a);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace

cudaError_t launch_w16_w13(const W16Args &a, cudaStream_t st) { return launch_w16<0>(a, st); }
cudaError_t launch_w16_w2(const W16Args &a, cudaStream_t st) { return launch_w16<1>(a, st); }

cudaError_t launch_gather_rows(const uint16_t *x, int H, int k, const int *row_src, const DevHeader *hdr,
                               int rows_cap, uint16_t *a, float *out, long long out_floats, cudaStream_t st)
{
    const long long warps = rows_cap > 0 ? rows_cap : 1;
    long long grid = (warps * 32 + 255) / 256;
    const long long cap = (long long)sm_count() * 8;
    if (grid > cap) grid = cap;
    const cudaError_t err = launch_pdl(gather_rows_kernel, dim3((int)grid), dim3(256), 0, st, x, H, k, row_src,
                                       hdr, a, reinterpret_cast<float4 *>(out), out_floats / 4);
    return err != cudaSuccess ? err : cudaGetLastError();
}

cudaError_t launch_prep_sf_w16(const uint8_t *sf, uint8_t *out, int E, int N, int K, cudaStream_t st)
{
    const long long groups = (long long)E * N / 64;
    const long long words = groups * (K / 64) * 64;
    long long grid = (words + 255) / 256;
    const long long cap = (long long)sm_count() * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    prep_sf_w16_kernel<<<(int)grid, 256, 0, st>>>(sf, out, groups, K);
    return cudaGetLastError();
}

}  // namespace nvfp4
