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
    int status;          // 0 = ok, 2 = a scale slot failed validation, 3 = bad expert id, 4 = prepared weights in
                         // the other scale format, 5 = device timeout
    int bad_count;       // number of bad scale slots
    int first_bad;       // lowest bad slot index (INT_MAX when none)
    int error_flags;     // kErr* bits below
    int num_mtiles;      // 128-row tiles of the padded permuted rows
    unsigned done_count; // CTAs of the routing histogram that finished
    int num_live_mtiles; // 128-row tiles holding at least one row (fewer than num_mtiles with 256-row padding)
    int pad[57];
};
static_assert(sizeof(DevHeader) == 256, "header is one 256-byte slot");

enum : int {
    kErrBadExpertId = 1,
    kErrTimeoutProducer = 2,
    kErrTimeoutMma = 4,
    kErrTimeoutEpilogue = 8,
    kErrTimeoutRoute = 16,
    kErrPlan = 32,  // a kernel was launched outside the conditions of its plan
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

// Packed FP32x2 arithmetic (one instruction, two IEEE round-to-nearest
// results) through the compiler's float2 builtins, so register pairs are
// allocated and scheduled like any other value; element 0 in .x.
typedef float2 f32x2;

__device__ __forceinline__ f32x2 pack_f32x2(float lo, float hi) { return make_float2(lo, hi); }
__device__ __forceinline__ f32x2 mul_f32x2(f32x2 a, f32x2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ f32x2 fma_f32x2(f32x2 a, f32x2 b, f32x2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float lo_f32(f32x2 v) { return v.x; }
__device__ __forceinline__ float hi_f32(f32x2 v) { return v.y; }

// Two BF16 values (one 32-bit word, element 0 in the low half) widened to FP32.
__device__ __forceinline__ f32x2 bf16x2_to_f32x2(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Four quotient pairs -> 32 bits of codes (pair i in byte i, the .x element
// of each pair in the low nibble).
__device__ __forceinline__ uint32_t e2m1_rn_sat8(f32x2 a, f32x2 b, f32x2 c, f32x2 d)
{
    uint32_t r;
    asm("{\n\t.reg .b8 ba, bb, bc, bd;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 ba, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 bb, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 bc, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 bd, %8, %7;\n\t"
        "mov.b32 %0, {ba, bb, bc, bd};\n\t}"
        : "=r"(r)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y), "f"(d.x), "f"(d.y));
    return r;
}

// The division table in the form the kernels keep in shared memory: the two
// constants of each E4M3 divisor duplicated into pairs, (zh, zh, zl, zl), and
// those of 6.
struct DivTable2 {
    float4 z[128];
    float2 six;
};
__device__ __forceinline__ void load_div_table(DivTable2 *dst, const DivTable &src)
{
    for (int i = threadIdx.x; i < 128; i += blockDim.x) {
        const float2 z = src.z[i];
        dst->z[i] = make_float4(z.x, z.x, z.y, z.y);
    }
    if (threadIdx.x == 0) dst->six = src.z[kE4M3Six];
}

// One 16-element block given as 8 pairs: returns the 64-bit packed codes
// (element i in nibble i) and writes the E4M3 scale byte.  `amax` is
// max |x_i|; `g` the global scale; `tab` the division table.
__device__ __forceinline__ uint2 quant_block16(const f32x2 (&x)[8], float amax, float g, const DivTable2 *tab,
                                               uint32_t &sf_byte)
{
    f32x2 q[8];
    const float ga = __fmul_rn(g, amax);
    uint32_t sb;
    if (ga <= kFltMax) {
        const float t = div_by_scale(ga, tab->six);  // fl(ga / 6)
        sb = e4m3_rn_sat(t);
        if (sb == 0) {
            sf_byte = 0;
            return make_uint2(0u, 0u);
        }
        const float4 z = tab->z[sb];  // (zh, zh, zl, zl)
        const f32x2 zh = make_float2(z.x, z.y), zl = make_float2(z.z, z.w);
        const f32x2 gg = pack_f32x2(g, g);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const f32x2 y = mul_f32x2(x[i], gg);
            q[i] = fma_f32x2(y, zh, mul_f32x2(y, zl));
        }
    } else {
        // g * amax overflowed: the scale saturates to 448 and the rare block
        // takes the plain IEEE division (infinite products stay infinite).
        sb = e4m3_rn_sat(__fdiv_rn(ga, 6.0f));
#pragma unroll
        for (int i = 0; i < 8; ++i)
            q[i] = pack_f32x2(__fdiv_rn(__fmul_rn(lo_f32(x[i]), g), 448.0f), __fdiv_rn(__fmul_rn(hi_f32(x[i]), g), 448.0f));
    }
    sf_byte = sb;
    return make_uint2(e2m1_rn_sat8(q[0], q[1], q[2], q[3]), e2m1_rn_sat8(q[4], q[5], q[6], q[7]));
}

// max |x| over 16 BF16 values in 8 words: signs cleared, the two halves
// compared as unsigned 16-bit integers (the magnitudes of non-negative
// floats order like their bit patterns), then the two halves.  As FP32.
__device__ __forceinline__ float amax16_bf16(const uint32_t *w)
{
    uint32_t m = w[0] & 0x7FFF7FFFu;
#pragma unroll
    for (int i = 1; i < 8; ++i) {
        const uint32_t v = w[i] & 0x7FFF7FFFu;
        asm("max.u16x2 %0, %0, %1;" : "+r"(m) : "r"(v));
    }
    return __uint_as_float(max(m << 16, m & 0xFFFF0000u));
}

// z * sigmoid(z) with the fast exponential and division (a few ulp; the
// requantisation that follows is exact for whatever FP32 h results).
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(fminf(-z, 80.0f))); }

// UE8M0 block scales.
// UE8M0 block scale of t >= 0 (t from the same fl(fl(g*amax)/6) as the E4M3
// path): the byte of the smallest power of two at or above t, clamped to the
// finite range 2^-127 .. 2^127 (bytes 0 .. 254).  Read off t's exponent field:
// a zero mantissa means t is itself a power of two.
__device__ __forceinline__ uint32_t ue8m0_round_up(float t)
{
    const uint32_t b = __float_as_uint(t);
    const uint32_t e = b >> 23, m = b & 0x7FFFFFu;
    if (e == 0) return m > 0x400000u ? 1u : 0u;  // subnormal t: 2^-127 covers up to 0x400000 * 2^-149
    const uint32_t c = e + (m != 0u ? 1u : 0u);
    return c > 254u ? 254u : c;                // also t = inf (e = 255)
}

// 1 / value(byte) = 2^(127 - byte), exact: a normal float for bytes 0 .. 253,
// the subnormal 2^-127 for byte 254.
__device__ __forceinline__ float ue8m0_reciprocal(uint32_t byte)
{
    return __uint_as_float(byte == 254u ? 0x00400000u : (254u - byte) << 23);
}

// quant_block16 with a UE8M0 block scale: the scale is t rounded up to a power
// of two, so fl(fl(x*g) / s) is one exact product by 1/s, rounded once.
__device__ __forceinline__ uint2 quant_block16_ue8m0(const f32x2 (&x)[8], float amax, float g, uint32_t &sf_byte)
{
    // fl(ga / 6) by the IEEE division: unlike the E4M3 path, the result matters
    // down to FP32 subnormals here
    const float t = __fdiv_rn(__fmul_rn(g, amax), 6.0f);
    const uint32_t sb = ue8m0_round_up(t);
    const float r = ue8m0_reciprocal(sb);
    const f32x2 gg = pack_f32x2(g, g), rr = pack_f32x2(r, r);
    f32x2 q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = mul_f32x2(mul_f32x2(x[i], gg), rr);
    sf_byte = sb;
    return make_uint2(e2m1_rn_sat8(q[0], q[1], q[2], q[3]), e2m1_rn_sat8(q[4], q[5], q[6], q[7]));
}

// UE8M0 scales carried to the tensor cores, one window per GEMM row.  The
// block-scaled FP4 MMA is given E4M3 scale bytes; its normal powers of two
// span 2^-6 .. 2^8 (15 binades, exponent fields 1 .. 15, mantissa 0).  Each
// operand row (a row of activations, or the weight row of one output column)
// carries its UE8M0 bytes b relative to its own largest byte m: with the
// row's shift c = max(m - 15, 0), byte b travels as the E4M3 byte with
// exponent field d = b - c, i.e. the value 2^(b - c - 7), when d lies in
// 1 .. 15, and as 0 when d <= 0 -- a block whose scale is more than 14
// binades below the row's largest (its values are below 2^-14 of the row's
// largest block).  The true scale is the carried one times 2^(c - 120), a
// power of two the GEMM epilogue multiplies back per row and per column: an
// exact product, so nothing depends on the global calibration and no scale is
// out of range.
__device__ __forceinline__ uint32_t ue8m0_row_shift(uint32_t row_max_byte)
{
    return row_max_byte > 15u ? row_max_byte - 15u : 0u;
}
// 2^(c - 120) for a row shift c in 0 .. 239 (a normal float).
__device__ __forceinline__ float ue8m0_row_factor(uint32_t c) { return __uint_as_float((c + 7u) << 23); }
// Row shift back from its factor.
__device__ __forceinline__ uint32_t ue8m0_shift_of_factor(float f) { return (__float_as_uint(f) >> 23) - 7u; }
// One byte carried with row shift c.  Bytes of a row never exceed its largest,
// so d <= 15; the mask only bounds the bytes of unused (padding) rows.
__device__ __forceinline__ uint32_t ue8m0_carried(uint32_t b, uint32_t c)
{
    const uint32_t d = b > c ? b - c : 0u;
    return (d & 15u) << 3;
}
// Four bytes (one 32-bit word) carried with the row shift c4 (c in every
// byte): a saturating byte-wise subtraction, then each 4-bit result moved to
// the exponent field (no byte overflows into its neighbour).
__device__ __forceinline__ uint32_t ue8m0_carried4(uint32_t w, uint32_t c4)
{
    return (__vsubus4(w, c4) & 0x0F0F0F0Fu) << 3;
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may be
// scheduled while its predecessor on the stream is still running: pdl_wait()
// blocks until the predecessor has completed and its memory is visible, and
// must come before anything it wrote is read.  pdl_trigger() lets the next
// kernel on the stream be scheduled once every CTA of this one has called it
// or exited.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Loads through L2 only (no L1 or texture-path copy), for the call's inputs
// that a kernel reads before its own pdl_wait (see the w13 GEMM's
// self-routed small-batch form).
__device__ __forceinline__ int ld_cg(const int *p)
{
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_cg(const float *p)
{
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_cg(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
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
