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
// of them), so each division uses two per-divisor constants and computes
// fma(y, zh, y * zl) -- the "division by a constant known in advance" of
// Brisebarre, Muller and Raina (IEEE Trans. Computers 53(8), 2004), here with
// zh = 1/s rounded toward zero and zl = RN(1/s - zh) >= 0.  With zl never
// negative a zero dividend keeps its sign ((-0)*zl + (-0)*zh = -0), so the
// quotient of -0 is -0 as IEEE division gives.  The host checks exhaustively
// that this equals the correctly rounded y/s for every E4M3 divisor and every
// FP32 significand (nvfp4_selftest_block_division); exponents only shift both
// sides, and results that leave the normal range are far below the smallest
// E2M1 step or saturate.  Two packed FP32x2 operations per pair of elements
// (plus the x*g product) replace two full IEEE divisions.
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

// Correctly rounded y / s for an E4M3 divisor with constants z = (zh, zl).
__device__ __forceinline__ float div_by_scale(float y, float2 z)
{
    return __fmaf_rn(y, z.x, __fmul_rn(y, z.y));
}

// Packed FP32x2 arithmetic (one instruction, two IEEE round-to-nearest results).
__device__ __forceinline__ float2 mul_f32x2(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pr;\n\tmov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "mul.rn.f32x2 pr, pa, pb;\n\tmov.b64 {%0, %1}, pr;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c)
{
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pc, pr;\n\tmov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "mov.b64 pc, {%6, %7};\n\tfma.rn.f32x2 pr, pa, pb, pc;\n\tmov.b64 {%0, %1}, pr;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

// Four quotient pairs -> 32 bits of codes (pair i in byte i, first element of
// each pair in the low nibble).
__device__ __forceinline__ uint32_t e2m1_rn_sat8(float2 a, float2 b, float2 c, float2 d)
{
    uint32_t r;
    asm("{\n\t.reg .b8 ba, bb, bc, bd;\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 ba, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 bb, %4, %3;\n\t"
        "mov.b16 lo, {ba, bb};\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 bc, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 bd, %8, %7;\n\t"
        "mov.b16 hi, {bc, bd};\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y), "f"(d.x), "f"(d.y));
    return r;
}

// One 16-element block given as 8 pairs: returns the 64-bit packed codes
// (element i in nibble i) and writes the E4M3 scale byte.  `amax` is
// max |x_i|; `g` the global scale; `tab` the division table.
__device__ __forceinline__ uint2 quant_block16(const float2 (&x)[8], float amax, float g, const float2 *tab,
                                               uint32_t &sf_byte)
{
    float2 q[8];
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
        const float2 gg = make_float2(g, g), zh = make_float2(z.x, z.x), zl = make_float2(z.y, z.y);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 y = mul_f32x2(x[i], gg);
            q[i] = fma_f32x2(y, zh, mul_f32x2(y, zl));
        }
    } else {
        // g * amax overflowed: the scale saturates to 448 and the rare block
        // takes the plain IEEE division (infinite products stay infinite).
        sb = e4m3_rn_sat(__fdiv_rn(ga, 6.0f));
#pragma unroll
        for (int i = 0; i < 8; ++i)
            q[i] = make_float2(__fdiv_rn(__fmul_rn(x[i].x, g), 448.0f), __fdiv_rn(__fmul_rn(x[i].y, g), 448.0f));
    }
    sf_byte = sb;
    return make_uint2(e2m1_rn_sat8(q[0], q[1], q[2], q[3]), e2m1_rn_sat8(q[4], q[5], q[6], q[7]));
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
