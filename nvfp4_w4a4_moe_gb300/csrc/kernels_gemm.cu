// Grouped block-scaled FP4 x FP4 expert GEMMs on the 5th-generation tensor
// cores (tcgen05, sm_103a), with the two fused epilogues of the MoE path.
//
// Page cited: "Gemma 4 NVFP4 MoE 空输出" (taking-lying-flat.github.io):
//   §矩阵融合 "MoE FFN": each expert gets M_e rows; the rows are reordered by
//   expert so all experts' GEMMs run as one grouped GEMM;
//   §矩阵融合 "Gated FFN": gate and up share the input and form one GEMM (w13),
//   followed by act(gate) * up and the down GEMM (w2);
//   §NVFP4 runtime-order figure: FP4 data + FP8 block scales enter the GEMM,
//   whose output scaling folds in both FP32 global scales;
//   pipeline figure: SiLU/mul + a2_gscale quantisation after w13, and the
//   token order restored and summed with the routing weights after w2.
//
// Kernel shape (one persistent CTA per SM, 10 warps):
//   warp 0     TMA producer: A tile 128 rows x 256 FP4 (128-byte swizzle),
//              B tile 128 rows x 256 FP4, and both 128x4-scale tiles (2 KB
//              each, plain bulk copies) per stage into a 6-stage (w13) or
//              5-stage (w2) ring.
//   warp 1     TMEM owner (512 columns) and MMA issuer: per stage, copies the
//              8 scale chunks smem -> TMEM (tcgen05.cp 32x128b.warpx4) and
//              issues 4 x tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X
//              (M128 N128 K64) into one of two FP32 accumulators.
//   warps 2-9  epilogue, two warps per TMEM lane quarter, each on half of the
//              tile's columns: tcgen05.ld of the accumulator, then either
//              SiLU(gate)*up + NVFP4 requantisation (w13) or the weighted
//              scatter-add into the token-order output (w2), transposed
//              through shared memory so the FP32 reductions are coalesced.
//              In the w13 kernel they first clear the output for w2.
// Every wait is bounded (%globaltimer); on expiry the kernel records the
// error in the workspace header, drains what it has in flight and exits.
#include <climits>

#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int BM = 128, BN = 128, BK = 256;  // BK in FP4 elements (128 bytes per row)
constexpr int A_BYTES = BM * BK / 2;
constexpr int B_BYTES = BN * BK / 2;
constexpr int SF_BYTES = 4 * 512;  // four 128x4-scale tiles = 256 K per stage
constexpr uint32_t TX_BYTES = A_BYTES + B_BYTES + 2 * SF_BYTES;
constexpr int ACC_COLS = BN;
constexpr int SF_TMEM_COL = 2 * ACC_COLS;  // 32 scale columns per stage after the accumulators
constexpr int TMEM_COLS = 512;
constexpr int NUM_EPI_WARPS = 8;  // two per TMEM lane quarter, each on half of the tile's columns
constexpr int EPI_THREADS = 32 * NUM_EPI_WARPS;
constexpr int COPY_WARP = 2 + NUM_EPI_WARPS;  // issues the smem -> TMEM scale copies
constexpr int NUM_THREADS = 64 + EPI_THREADS + 32;
constexpr int XPOSE_LD = 33;  // padded row of the per-warp 32 x 32 transpose buffer
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;

// Shared-memory plan per kernel: the w13 kernel spends it all on a 6-stage
// ring (the loads of a stage take longer than its MMAs, so more bytes in
// flight hide more latency); the w2 kernel keeps 5 stages and a transpose
// buffer for its epilogue.
#ifndef NVFP4_W13_STAGES
#define NVFP4_W13_STAGES 6
#endif
template <int EPI>
struct Plan {
    static constexpr int STAGES = EPI == 0 ? NVFP4_W13_STAGES : 5;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SF_BYTES;
    static constexpr int OFF_BAR = OFF_SFB + STAGES * SF_BYTES;
    static constexpr int NUM_BARS = 3 * STAGES + 4 + 2;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_XPOSE = (OFF_MISC + 16 + 15) & ~15;
    static constexpr int XPOSE_BYTES = EPI == 1 ? NUM_EPI_WARPS * 32 * XPOSE_LD * 4 : 0;
    static constexpr int SMEM_BYTES = OFF_XPOSE + XPOSE_BYTES + 1024;  // + alignment slack
    static_assert(SF_TMEM_COL + STAGES * 32 <= TMEM_COLS, "scale slots exceed TMEM");
    static_assert(SMEM_BYTES + 1024 <= 232448, "shared memory plan exceeds the opt-in limit");
};

// Instruction descriptor, block-scaled kinds: E2M1 A and B (code 1 at bits
// 7-9 and 10-12), K-major both, N>>3 at 17-22, scale type UE4M3 (bit 23 = 0),
// M>>4 at 24-28, scale-factor ids 0.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t *b, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase of parity `parity`; false on expiry or abort.
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, volatile int *abort_flag,
                                          uint64_t limit)
{
    if (mbar_test(b, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_test(b, parity)) return true;
        if (abort_flag && *abort_flag) return false;
        if (global_timer_ns() - t0 > limit) return false;
    }
}

// ---------------------------------------------------------------- copies
__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     su32(dst)),
                 "l"(src), "r"(bytes), "r"(su32(bar))
                 : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
                 : "memory");
}
// K-major operand tile, 128-byte swizzle: 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// One 128x4-scale tile as 32 rows x 16 bytes, no swizzle (8-row groups 128 B apart).
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d),
        "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v)
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// z * sigmoid(z) with the fast exponential and division (a few ulp; the
// requantisation that follows is exact for whatever FP32 h results).
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(fminf(-z, 80.0f))); }

// ---------------------------------------------------------------- kernel
template <int EPI>  // 0: w13 (SiLU*up + requantise), 1: w2 (weighted combine)
__global__ void __launch_bounds__(NUM_THREADS, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const GemmArgs p, const DivTable tab_in)
{
    using P = Plan<EPI>;
    constexpr int STAGES = P::STAGES, OFF_A = P::OFF_A, OFF_B = P::OFF_B, OFF_SFA = P::OFF_SFA,
                  OFF_SFB = P::OFF_SFB, OFF_BAR = P::OFF_BAR, OFF_MISC = P::OFF_MISC, OFF_XPOSE = P::OFF_XPOSE;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ DivTable2 tab;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *full = bars, *empty = bars + STAGES, *acc_full = bars + 2 * STAGES,
             *acc_empty = bars + 2 * STAGES + 2, *drain = bars + 2 * STAGES + 4, *sf_ready = bars + 2 * STAGES + 5,
             *drain_cp = bars + 3 * STAGES + 5;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (p.hdr->status != 0) return;
    const int NT = p.N / BN;
    const int ntiles = p.hdr->num_mtiles * NT;
    if ((int)blockIdx.x >= ntiles) return;
    const int KT = (p.K + BK - 1) / BK;

    if (EPI == 0) load_div_table(&tab, tab_in);
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_ready[s], 1);
        }
        mbar_init(drain_cp, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], EPI_THREADS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t stage = 0, phase = 0;
        uint32_t issued = 0;           // bit s: stage s has had a load issued
        uint32_t last_parity = 0;      // bit s: parity of that last load's phase
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            const int mt = tile / NT, nt = tile - mt * NT;
            const int e = p.tile_expert[mt];
            for (int kt = 0; kt < KT; ++kt) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                uint64_t *fb = &full[stage];
                mbar_expect_tx(fb, TX_BYTES);
                const int kx = kt * (BK / 2);
                uint8_t *sa = smem + OFF_A + stage * A_BYTES;
                uint8_t *sb = smem + OFF_B + stage * B_BYTES;
                tma_2d(sa, &tmap_a, kx, mt * BM, fb);
                if (p.gate_up_I > 0) {
                    const int brow = e * 2 * p.gate_up_I + nt * 64;
                    tma_2d(sb, &tmap_b, kx, brow, fb);
                    tma_2d(sb + B_BYTES / 2, &tmap_b, kx, brow + p.gate_up_I, fb);
                } else {
                    tma_2d(sb, &tmap_b, kx, e * p.N + nt * BN, fb);
                }
                bulk_g2s(smem + OFF_SFA + stage * SF_BYTES, p.a_sf + ((size_t)mt * p.a_kc + 4 * kt) * 512,
                         SF_BYTES, fb);
                bulk_g2s(smem + OFF_SFB + stage * SF_BYTES,
                         p.b_sf + (((size_t)e * NT + nt) * p.b_kc + 4 * kt) * 512, SF_BYTES, fb);
                issued |= 1u << stage;
                last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            atomicOr(&p.hdr->error_flags, kErrTimeoutProducer);
        }
        // Drain: every issued load has landed before the CTA exits.
        for (int s = 0; s < STAGES; ++s)
            if (issued & (1u << s)) mbar_wait(&full[s], (last_parity >> s) & 1u, nullptr, kDrainLimitNs);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + acc * ACC_COLS;
            for (int kt = 0; kt < KT; ++kt) {
                // operands landed (full) and their scales are in TMEM (sf_ready)
                if (!mbar_wait(&full[stage], phase, abort_flag, kWaitLimitNs) ||
                    !mbar_wait(&sf_ready[stage], phase, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int ksteps = min(4, (p.K - kt * BK + 63) / 64);
                const uint32_t sfa_t = tmem + SF_TMEM_COL + stage * 32, sfb_t = sfa_t + 16;
                const uint32_t sa = su32(smem + OFF_A + stage * A_BYTES);
                const uint32_t sb = su32(smem + OFF_B + stage * B_BYTES);
                for (int j = 0; j < ksteps; ++j)
                    tc_mma(d, desc_sw128(sa + 32 * j), desc_sw128(sb + 32 * j), sfa_t + 4 * j, sfb_t + 4 * j,
                           (kt | j) != 0);
                tc_commit(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            tc_commit(&acc_full[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (!ok) {
            *abort_flag = 1;
            atomicOr(&p.hdr->error_flags, kErrTimeoutMma);
        }
        // Drain: all issued tcgen05 work completes before TMEM is released.
        tc_commit(drain);
        mbar_wait(drain, 0, nullptr, kDrainLimitNs);
    } else if (warp == COPY_WARP && lane == 0) {
        // ------------------------------------------------ scale copier
        // Moves each stage's scale tiles smem -> TMEM (tcgen05.cp
        // 32x128b.warpx4, one per K step and operand) ahead of the MMA issuer,
        // and signals sf_ready[stage] when the copies have completed.  The
        // stage's TMEM scale slot is only rewritten after the producer has
        // refilled the stage, i.e. after the MMAs that read it have finished.
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            for (int kt = 0; kt < KT; ++kt) {
                if (!mbar_wait(&full[stage], phase, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int ksteps = min(4, (p.K - kt * BK + 63) / 64);
                const uint32_t sfa_t = tmem + SF_TMEM_COL + stage * 32, sfb_t = sfa_t + 16;
                const uint32_t ssfa = su32(smem + OFF_SFA + stage * SF_BYTES);
                const uint32_t ssfb = su32(smem + OFF_SFB + stage * SF_BYTES);
                for (int j = 0; j < ksteps; ++j) {
                    tc_cp_sf(sfa_t + 4 * j, desc_sf(ssfa + 512 * j));
                    tc_cp_sf(sfb_t + 4 * j, desc_sf(ssfb + 512 * j));
                }
                tc_commit(&sf_ready[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            atomicOr(&p.hdr->error_flags, kErrTimeoutMma);
        }
        tc_commit(drain_cp);
        mbar_wait(drain_cp, 0, nullptr, kDrainLimitNs);
    } else if (warp >= 2 && warp < COPY_WARP) {
        // ------------------------------------------------ epilogue
        const int ew = warp - 2;          // 0..7
        const int quarter = warp & 3;     // TMEM lanes this warp may read
        const int half = ew >> 2;         // which half of the tile's columns it owns
        const int r_in = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        if (EPI == 0 && p.zero_out) {
            // Clear the FP32 output for the w2 kernel's reductions while the
            // first accumulator is being produced.
            const long long active = min((long long)gridDim.x, (long long)ntiles);
            const long long n4 = p.zero_floats >> 2;
            float4 *z = reinterpret_cast<float4 *>(p.zero_out);
            for (long long i = (long long)blockIdx.x * EPI_THREADS + (threadIdx.x - 64); i < n4;
                 i += active * EPI_THREADS)
                z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float *xp = reinterpret_cast<float *>(smem + OFF_XPOSE) + ew * 32 * XPOSE_LD;
        uint32_t acc = 0, acc_phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            const int mt = tile / NT, nt = tile - mt * NT;
            const int e = p.tile_expert[mt];
            const int row = mt * BM + r_in;
            const bool valid = row < p.pad_off[e] + p.counts[e];
            if (!mbar_wait(&acc_full[acc], acc_phase, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t col0 = lane_base + acc * ACC_COLS;
            if (EPI == 0) {
                // SiLU(gate) * up on this warp's 32 of the tile's 64 h columns
                // (gate columns 0..63 of the tile, up columns 64..127), then the
                // a2 quantisation of the result, 16 columns per block.
                const float alpha = p.alpha[e], g2 = p.g2[e];
                const f32x2 aa = pack_f32x2(alpha, alpha);
                uint32_t sfw = 0;
#pragma unroll 1
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int c = half * 2 + c2;
                    float gate[16], up[16];
                    tmem_ld16(col0 + 16 * c, gate);
                    tmem_ld16(col0 + 64 + 16 * c, up);
                    tmem_wait_ld();
                    f32x2 h[8];
                    float amax = 0.0f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const f32x2 gs = mul_f32x2(pack_f32x2(gate[2 * i], gate[2 * i + 1]), aa);
                        const f32x2 us = mul_f32x2(pack_f32x2(up[2 * i], up[2 * i + 1]), aa);
                        h[i] = mul_f32x2(pack_f32x2(silu(lo_f32(gs)), silu(hi_f32(gs))), us);
                        amax = fmaxf(amax, fmaxf(fabsf(lo_f32(h[i])), fabsf(hi_f32(h[i]))));
                    }
                    if (p.h_dump && valid) {
                        float4 *hd = reinterpret_cast<float4 *>(p.h_dump + (size_t)row * p.I + nt * 64 + 16 * c);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            hd[i] = make_float4(lo_f32(h[2 * i]), hi_f32(h[2 * i]), lo_f32(h[2 * i + 1]), hi_f32(h[2 * i + 1]));
                    }
                    uint32_t sb;
                    const uint2 pk = quant_block16(h, amax, g2, &tab, sb);
                    if (valid) *reinterpret_cast<uint2 *>(p.a2q + (size_t)row * (p.I >> 1) + nt * 32 + 8 * c) = pk;
                    sfw |= sb << (8 * c2);
                }
                if (valid) {
                    *reinterpret_cast<uint16_t *>(p.sf2 + swz_sf_offset(row, nt, p.kc2) + 2 * half) = (uint16_t)sfw;
                    if (nt == NT - 1 && half == 0)
                        for (int cc = NT; cc < p.kc2; ++cc)
                            *reinterpret_cast<uint32_t *>(p.sf2 + swz_sf_offset(row, cc, p.kc2)) = 0u;
                }
            } else {
                // out[t, cols] += w[t, j] * alpha2 * y2: this warp's 64 columns,
                // 32 at a time, transposed through shared memory so that each
                // reduction instruction covers four contiguous 128-byte row
                // segments.
                int t = 0;
                float scale = 0.0f;
                if (valid) {
                    const int f = p.row_src[row];
                    t = f / p.k;
                    scale = __fmul_rn(p.topk_w[f], p.alpha[e]);
                }
                const int sub = lane >> 3, cc = (lane & 7) * 4;
#pragma unroll 1
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int cbase = 64 * half + 32 * c2;
                    float v[32];
                    tmem_ld16(col0 + cbase, v);
                    tmem_ld16(col0 + cbase + 16, v + 16);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) xp[lane * XPOSE_LD + i] = v[i] * scale;
                    __syncwarp();
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int rr = it * 4 + sub;
                        const int t_r = __shfl_sync(0xffffffffu, t, rr);
                        const int ok_r = __shfl_sync(0xffffffffu, (int)valid, rr);
                        const float *src = xp + rr * XPOSE_LD + cc;
                        if (ok_r)
                            red_add_v4(p.out + (size_t)t_r * p.H + nt * BN + cbase + cc, src[0], src[1], src[2], src[3]);
                    }
                    __syncwarp();
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
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
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D byte tensor [rows, row_bytes] with a (128 bytes x box_rows) box, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d) for a %llu x %llu byte tensor", (int)r,
                  (unsigned long long)rows, (unsigned long long)row_bytes);
        return false;
    }
    return true;
}

template <int EPI>
cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t st)
{
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t err = cudaFuncSetAttribute(moe_gemm_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               Plan<EPI>::SMEM_BYTES);
        if (err != cudaSuccess) return err;
        attr_set = true;
    }
    CUtensorMap ma, mb;
    const uint64_t kbytes = (uint64_t)a.K / 2;
    if (!make_map(&ma, a.a_q, kbytes, (uint64_t)a.rows_cap, 128)) return cudaErrorInvalidValue;
    const uint64_t brows = (uint64_t)a.E * (uint64_t)a.N;
    if (!make_map(&mb, a.b_q, kbytes, brows, a.gate_up_I > 0 ? 64 : 128)) return cudaErrorInvalidValue;
    const long long tiles = (long long)a.mtiles_cap * (a.N / BN);
    int grid = sm_count();
    if (tiles < grid) grid = (int)(tiles > 0 ? tiles : 1);
    moe_gemm_kernel<EPI><<<grid, NUM_THREADS, Plan<EPI>::SMEM_BYTES, st>>>(ma, mb, a, div_table());
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_w13(const GemmArgs &a, cudaStream_t st) { return launch_gemm<0>(a, st); }
cudaError_t launch_gemm_w2(const GemmArgs &a, cudaStream_t st) { return launch_gemm<1>(a, st); }

}  // namespace nvfp4
