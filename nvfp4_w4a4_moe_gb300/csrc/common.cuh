// Device-side helpers shared by the NVFP4 MoE kernels (sm_103a).
//
// The activation quantisation follows the page "Gemma 4 NVFP4 MoE 空输出"
// (§NVFP4, runtime-order figure): per 16-element block,
//     s = e4m3( fl(fl(g * amax) / 6) ),   q_i = e2m1( fl(fl(x_i * g) / s) ),
// with the hardware round-to-nearest-even, saturating conversions
// cvt.rn.satfinite.{e4m3x2,e2m1x2}.f32 that the page names.
//
// Exact division by a block scale.  Both divisions above must be the correctly
// rounded FP32 quotient.  The divisor s is one of 126 E4M3 values (and 6 is one
// of them), so each division uses two per-divisor constants zh = RN(1/s) and
// zl = RN(1/s - zh) and computes fma(y, zh, y * zl) -- the "division by a
// constant known in advance" of Brisebarre, Muller and Raina (IEEE Trans.
// Computers 53(8), 2004).  The host checks exhaustively that this equals the
// correctly rounded y/s for every E4M3 divisor and every FP32 significand
// (nvfp4_selftest_block_division); exponents only shift both sides, and
// results that leave the normal range are far below the smallest E2M1 step or
// saturate; zero dividends keep their sign.  One FMUL, one FFMA and a sign
// copy replace a full IEEE division per element.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

// (zh, zl) per E4M3 byte; byte 0 (scale 0) is never divided by.
struct DivTable {
    float2 z[128];
};

constexpr int kE4M3Six = 0x4C;  // E4M3 byte of 6.0 (the E2M1 maximum)
constexpr float kFltMax = 3.40282346638528859812e+38f;

// Device-side status block at the start of every workspace.
struct DevHeader {
    int status;          // 0 = ok, 2 = a scale slot failed validation, 3 = bad expert id
    int bad_count;       // number of bad scale slots
    int first_bad;       // lowest bad slot index (INT_MAX when none)
    int error_flags;     // kErr* bits below
    int num_mtiles;      // 128-row tiles of the padded permuted rows
    unsigned done_count; // CTAs of the routing histogram that finished
    int pad[58];
};
static_assert(sizeof(DevHeader) == 256, "header is one 256-byte slot");

enum : int {
    kErrBadExpertId = 1,
    kErrTimeoutProducer = 2,
    kErrTimeoutMma = 4,
    kErrTimeoutEpilogue = 8,
};

// RN, saturating FP32 -> E4M3 (t >= 0): the byte of the second source.
__device__ __forceinline__ uint32_t e4m3_rn_sat(float t)
{
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
    return (uint32_t)r & 0xFFu;
}

// RN, saturating FP32 -> E2M1 for four values: a in bits 0-3, b in 4-7,
// c in 8-11, d in 12-15 (the x2 conversion puts its first source in the upper
// nibble, so the pair (a, b) is passed as (b, a)).
__device__ __forceinline__ uint32_t e2m1_rn_sat4(float a, float b, float c, float d)
{
    uint32_t r;
    asm("{\n\t.reg .b8 ab, cd;\n\t.reg .b16 w;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 ab, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 cd, %4, %3;\n\t"
        "mov.b16 w, {ab, cd};\n\t"
        "cvt.u32.u16 %0, w;\n\t}"
        : "=r"(r)
        : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}

// Correctly rounded y / s for an E4M3 divisor with constants z = (zh, zl).
// The two-constant form loses the sign of a zero dividend when zl < 0
// ((-0)*zl = +0, and -0 + +0 = +0); the quotient always has the dividend's
// sign, so it is put back.
__device__ __forceinline__ float div_by_scale(float y, float2 z)
{
    return copysignf(__fmaf_rn(y, z.x, __fmul_rn(y, z.y)), y);
}

// One 16-element block: returns the 64-bit packed codes (element i in nibble
// i) and writes the E4M3 scale byte.  `amax` is max |x_i|; `g` the global
// scale; `tab` the division table (any address space).
__device__ __forceinline__ uint2 quant_block16(const float (&x)[16], float amax, float g,
                                               const float2 *tab, uint32_t &sf_byte)
{
    float q[16];
    const float ga = __fmul_rn(g, amax);
    uint32_t sb;
    if (ga <= kFltMax) {
        const float t = div_by_scale(ga, tab[kE4M3Six]);  // fl(ga / 6)
        sb = e4m3_rn_sat(t);
        if (sb == 0) {
            sf_byte = 0;
            return make_uint2(0u, 0u);
        }
        const float2 z = tab[sb];
#pragma unroll
        for (int i = 0; i < 16; ++i) q[i] = div_by_scale(__fmul_rn(x[i], g), z);
    } else {
        // g * amax overflowed: the scale saturates to 448 and the rare block
        // takes the plain IEEE division (infinite products stay infinite).
        sb = e4m3_rn_sat(__fdiv_rn(ga, 6.0f));
        const float s = 448.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) q[i] = __fdiv_rn(__fmul_rn(x[i], g), s);
    }
    sf_byte = sb;
    uint2 r;
    r.x = e2m1_rn_sat4(q[0], q[1], q[2], q[3]) | (e2m1_rn_sat4(q[4], q[5], q[6], q[7]) << 16);
    r.y = e2m1_rn_sat4(q[8], q[9], q[10], q[11]) | (e2m1_rn_sat4(q[12], q[13], q[14], q[15]) << 16);
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Byte offset of (row, 64-element column chunk) in the swizzled scale layout
// with `kc` chunks per 128-row tile; the four scales of the chunk follow.
__device__ __forceinline__ size_t swz_sf_offset(int row, int chunk, int kc)
{
    return ((size_t)(row >> 7) * kc + chunk) * 512 + (size_t)(row & 31) * 16 + ((row >> 5) & 3) * 4;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace nvfp4
