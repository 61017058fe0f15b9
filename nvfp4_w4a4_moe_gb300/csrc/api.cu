// C ABI of libnvfp4moe: argument checks, workspace layout and the launch
// sequence of the NVFP4 MoE expert path.  Declared in include/nvfp4_moe.h.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include "../../include/nvfp4_moe.h"
#include "internal.h"

namespace nvfp4 {

// ------------------------------------------------------------------ errors
static thread_local char g_err[512] = "no error";

void set_error(const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
}

static int fail(int status, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return status;
}

static int cuda_fail(cudaError_t e, const char *what)
{
    return fail(NVFP4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define NV_CUDA(call, what)                                  \
    do {                                                     \
        cudaError_t _e = (call);                             \
        if (_e != cudaSuccess) return cuda_fail(_e, (what)); \
    } while (0)

// ------------------------------------------------------------------ device facts
int sm_count()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

// ------------------------------------------------------------------ block-scale division table
static double e4m3_value(int b)
{
    const int e = (b >> 3) & 15, m = b & 7;
    return e == 0 ? std::ldexp((double)m, -9) : std::ldexp(8.0 + m, e - 10);
}

// zh = 1/s rounded toward zero, zl = RN(1/s - zh) >= 0, for each finite
// non-zero E4M3 scale s (two-constant division; see common.cuh).
static DivTable build_div_table()
{
    DivTable t;
    std::memset(&t, 0, sizeof(t));
    for (int b = 1; b <= 0x7E; ++b) {
        const double s = e4m3_value(b);
        const double r = 1.0 / s;  // 1/s = m * 2^e with m a short odd fraction; r is its nearest double
        float zh = (float)r;
        if ((double)zh > r) zh = std::nextafterf(zh, 0.0f);
        const double rem = std::fma(-s, (double)zh, 1.0);  // exact: 1 - s*zh >= 0
        const float zl = (float)(rem / s);
        t.z[b] = make_float2(zh, zl);
    }
    return t;
}

const DivTable &div_table()
{
    static const DivTable t = build_div_table();
    return t;
}

// ------------------------------------------------------------------ workspace layout
static size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

WsLayout make_layout(int T, int H, int I, int E, int k)
{
    WsLayout L;
    std::memset(&L, 0, sizeof(L));
    L.T = T, L.H = H, L.I = I, L.E = E, L.k = k;
    L.R = T * k;
    const long long R = L.R;
    // rows padded per expert to 256 (the paired w13 GEMM) at most: every busy
    // expert may end on a partial 256-row block
    const long long busy = R < E ? R : E;
    L.rows_cap = R == 0 ? 0 : (int)(((R + busy * 255) + 255) / 256 * 256);
    L.mtiles_cap = L.rows_cap / 128;
    L.nchunks = (int)((R + kRouteChunk - 1) / kRouteChunk);
    if (L.nchunks < 1) L.nchunks = 1;
    L.kc1 = 4 * ((H + 255) / 256);
    L.kc2 = 4 * ((I + 255) / 256);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = up256(o + bytes);
        return at;
    };
    L.hdr = take(sizeof(DevHeader));
    L.g1 = take(sizeof(float) * 4 * (size_t)E);  // g1, g2, gw13, gw2
    L.g2 = L.g1 + sizeof(float) * (size_t)E;
    L.alpha1 = take(sizeof(float) * 2 * (size_t)E);
    L.alpha2 = L.alpha1 + sizeof(float) * (size_t)E;
    L.counts = take(sizeof(int) * (size_t)E);
    L.offsets = take(sizeof(int) * (size_t)(E + 1));
    L.pad_off = take(sizeof(int) * (size_t)(E + 1));
    L.chunk_hist = take(sizeof(int) * (size_t)L.nchunks * E);
    L.row_of = take(sizeof(int) * (size_t)R);
    L.perm = take(sizeof(int) * (size_t)R);
    L.row_src = take(sizeof(int) * (size_t)L.rows_cap);
    L.tile_expert = take(sizeof(int) * (size_t)L.mtiles_cap);
    L.live_mtiles = take(sizeof(int) * (size_t)L.mtiles_cap);
    L.row_max = take(sizeof(int) * 2 * (size_t)L.rows_cap);  // UE8M0: a1 rows, then a2 rows
    L.a1q = take((size_t)L.rows_cap * (H / 2));
    L.sf1 = take((size_t)L.mtiles_cap * L.kc1 * 512);
    L.a2q = take((size_t)L.rows_cap * (I / 2));
    L.sf2 = take((size_t)L.mtiles_cap * L.kc2 * 512);
    L.end = o;
    L.x_stage = take(sizeof(uint16_t) * (size_t)T * H);
    L.ids_stage = take(sizeof(int32_t) * (size_t)R);
    L.w_stage = take(sizeof(float) * (size_t)R);
    L.out_stage = take(sizeof(float) * (size_t)T * H);
    L.status_stage = take(sizeof(DevHeader) * (size_t)kMaxHostChunks);
    L.host_end = o;
    return L;
}

static size_t prepared_w13_bytes(int E, int H, int I)
{
    return (size_t)E * (2 * I / 128) * (4 * ((H + 255) / 256)) * 512;
}
static size_t prepared_w2_bytes(int E, int H, int I)
{
    return (size_t)E * (H / 128) * (4 * ((I + 255) / 256)) * 512;
}

static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The activation quantiser addresses its outputs with 32-bit offsets: scale
// bytes (both layouts, rows rounded up to 128) must stay below 2^32.
static bool quant_offsets_fit(long long rows, int H)
{
    const long long kc = (H + 63) / 64;
    return ((rows + 127) / 128) * kc * 512 < (1ll << 32);
}

int quantize_shape_status(int T, int H, int k, int E)
{
    if (E < 1 || E > 1024 || k < 1 || k > 32 || k > E || T < 0)
        return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "quantize: E=%d k=%d T=%d unsupported", E, k, T);
    if (H <= 0 || H % 64 != 0) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "quantize: H=%d is not a multiple of 64", H);
    if (!quant_offsets_fit((long long)T * k, H))
        return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "quantize: T*k*H/16 = %lld scale bytes exceed 2^32",
                    (long long)T * k * (H / 16));
    return NVFP4_OK;
}

static int check_layer_shape(int E, int H, int I, int k)
{
    if (E < 1 || E > 1024) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "E=%d outside [1, 1024]", E);
    if (k < 1 || k > 32 || k > E) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "k=%d outside [1, min(32, E)]", k);
    if (H <= 0 || H % 256 != 0) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "H=%d is not a positive multiple of 256", H);
    if (I <= 0 || I % 64 != 0) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "I=%d is not a positive multiple of 64", I);
    return NVFP4_OK;
}

static int read_header(const void *ws, cudaStream_t st, DevHeader *h)
{
    NV_CUDA(cudaMemcpyAsync(h, ws, sizeof(DevHeader), cudaMemcpyDeviceToHost, st), "reading the status block");
    NV_CUDA(cudaStreamSynchronize(st), "synchronising the stream");
    return NVFP4_OK;
}

static int header_status(const DevHeader &h, int *first_bad)
{
    if (first_bad) *first_bad = h.first_bad == 0x7fffffff ? -1 : h.first_bad;
    if (h.status == 2)
        return fail(NVFP4_ERR_SCALE_INVALID, "%d scale slot(s) failed validation; first bad slot %d", h.bad_count,
                    h.first_bad);
    if (h.status == 3 || (h.error_flags & kErrBadExpertId))
        return fail(NVFP4_ERR_INVALID_ARG, "an expert id is outside [0, E)");
    if (h.status == 4)
        return fail(NVFP4_ERR_INVALID_ARG, "the prepared weights were converted for the other block-scale format");
    if (h.status == 5 || (h.error_flags & (kErrTimeoutProducer | kErrTimeoutMma | kErrTimeoutEpilogue | kErrTimeoutRoute)))
        return fail(NVFP4_ERR_DEVICE_TIMEOUT, "a device-side wait expired (flags 0x%x)", h.error_flags);
    if (h.error_flags & kErrPlan)
        return fail(NVFP4_ERR_CUDA, "a GEMM was launched outside its plan's conditions (flags 0x%x)", h.error_flags);
    return NVFP4_OK;
}

// ------------------------------------------------------------------ self-test of the division
long long selftest_division(int nthreads)
{
    const DivTable &t = div_table();
    if (nthreads <= 0) nthreads = (int)std::thread::hardware_concurrency();
    if (nthreads <= 0) nthreads = 1;
    std::atomic<long long> bad{0};
    std::atomic<int> next{1};
    auto work = [&]() {
        for (;;) {
            const int b = next.fetch_add(1);
            if (b > 0x7E) return;
            const double s = e4m3_value(b);
            // s = D * 2^es with D odd
            int es = 0;
            double D = s;
            while (D != std::floor(D)) D *= 2, --es;
            while (std::fmod(D, 2.0) == 0.0) D /= 2, ++es;
            const uint64_t d = (uint64_t)D;
            const float zh = t.z[b].x, zl = t.z[b].y;
            long long local = 0;
            for (uint32_t Y = 1u << 23; Y < (1u << 24); ++Y) {
                const float y = std::ldexp((float)Y, -23);
                volatile float prod = y * zl;  // one rounding, no contraction
                const float q = std::fmaf(y, zh, prod);
                int sh = 0;
                while ((((uint64_t)Y << sh) / d) < (1u << 23)) ++sh;
                const uint64_t N = (uint64_t)Y << sh;
                uint64_t Q = N / d;
                const uint64_t R = N % d;
                if (2 * R > d || (2 * R == d && (Q & 1))) ++Q;
                const double want = std::ldexp((double)Q, -sh - 23 - es);
                if ((double)q != want) ++local;
            }
            bad += local;
        }
    };
    std::vector<std::thread> pool;
    for (int i = 0; i < nthreads; ++i) pool.emplace_back(work);
    for (auto &th : pool) th.join();
    return bad.load();
}

}  // namespace nvfp4

using namespace nvfp4;

// ====================================================================== C ABI
extern "C" {

const char *nvfp4_last_error_string(void) { return g_err; }

int nvfp4_version(void) { return 100; }

long long nvfp4_selftest_block_division(int nthreads) { return selftest_division(nthreads); }

int nvfp4_selftest_ue8m0_carry(uint8_t *out, nvfp4_stream_t stream)
{
    if (!out) return fail(NVFP4_ERR_INVALID_ARG, "selftest: out is null");
    if (!aligned(out, 4)) return fail(NVFP4_ERR_INVALID_ARG, "selftest: out must be 4-byte aligned");
    cudaStream_t st = (cudaStream_t)stream;
    NV_CUDA(launch_ue8m0_carry_selftest(out, st), "launching the carry self-test");
    NV_CUDA(cudaStreamSynchronize(st), "synchronising the stream");
    return NVFP4_OK;
}

int nvfp4_selftest_device_wait(void *ws, size_t ws_bytes, unsigned limit_us, nvfp4_stream_t stream)
{
    if (!ws || !aligned(ws, 256) || ws_bytes < sizeof(DevHeader))
        return fail(NVFP4_ERR_INVALID_ARG, "selftest: workspace null, misaligned or below 256 bytes");
    if (limit_us == 0 || limit_us > 1000000u)
        return fail(NVFP4_ERR_INVALID_ARG, "selftest: limit %u us outside [1, 10^6]", limit_us);
    cudaStream_t st = (cudaStream_t)stream;
    NV_CUDA(cudaMemsetAsync(ws, 0, sizeof(DevHeader), st), "clearing the status block");
    NV_CUDA(launch_wait_selftest(static_cast<DevHeader *>(ws), (uint64_t)limit_us * 1000u, st),
            "launching the wait self-test");
    return NVFP4_OK;
}

int nvfp4_validate_scales(const float *scales, const uint8_t *written, int n, void *ws, nvfp4_stream_t stream,
                          int *bad_count_host, int *first_bad_host)
{
    if (n < 0 || !bad_count_host || !first_bad_host || !ws || (n > 0 && !scales))
        return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_validate_scales: bad arguments");
    if (!aligned(ws, 256)) return fail(NVFP4_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
    cudaStream_t st = (cudaStream_t)stream;
    DevHeader *hdr = reinterpret_cast<DevHeader *>(ws);
    ValidateArgs va;
    std::memset(&va, 0, sizeof(va));
    va.s[0] = scales;
    va.written[0] = written;
    va.E = n;
    va.narrays = 1;
    va.hdr = hdr;
    NV_CUDA(launch_validate(va, st), "launching the scale check");
    DevHeader h;
    int rc = read_header(ws, st, &h);
    if (rc) return rc;
    *bad_count_host = h.bad_count;
    *first_bad_host = h.bad_count ? h.first_bad : -1;
    return NVFP4_OK;
}

size_t nvfp4_quantize_workspace_size(int T, int k, int E)
{
    if (T < 0 || k < 1 || E < 1 || (long long)T * k > INT_MAX) return 0;
    return make_layout(T, 256, 64, E, k).row_src;  // header .. perm
}

int nvfp4_quantize_experts(const uint16_t *x, int T, int H, const int32_t *topk_ids, int k, int E,
                           const float *input_scale, uint8_t *q_out, uint8_t *sf_out, int sf_layout,
                           int32_t *expert_offsets, int32_t *perm, void *ws, size_t ws_bytes,
                           nvfp4_stream_t stream)
{
    const int shape_rc = quantize_shape_status(T, H, k, E);
    if (shape_rc != NVFP4_OK) return shape_rc;
    const int sf_ue8m0 = (sf_layout & NVFP4_SF_UE8M0) != 0;
    sf_layout &= ~NVFP4_SF_UE8M0;
    if (sf_layout != NVFP4_SF_LINEAR && sf_layout != NVFP4_SF_SWIZZLED)
        return fail(NVFP4_ERR_INVALID_ARG, "unknown scale layout %d", sf_layout);
    if (!input_scale || !expert_offsets || !ws || (T > 0 && (!x || !topk_ids || !q_out || !sf_out || !perm)))
        return fail(NVFP4_ERR_INVALID_ARG, "quantize: null pointer");
    if (!aligned(ws, 256) || (T > 0 && (!aligned(x, 16) || !aligned(q_out, 16) || !aligned(sf_out, 4))))
        return fail(NVFP4_ERR_INVALID_ARG, "quantize: misaligned pointer (x 16 B, q 16 B, sf 4 B, ws 256 B)");
    const size_t need = nvfp4_quantize_workspace_size(T, k, E);
    if (ws_bytes < need) return fail(NVFP4_ERR_WORKSPACE_TOO_SMALL, "quantize: workspace %zu < %zu", ws_bytes, need);
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t *base = static_cast<uint8_t *>(ws);
    WsLayout L = make_layout(T, 256, 64, E, k);
    DevHeader *hdr = reinterpret_cast<DevHeader *>(base + L.hdr);
    float *g = reinterpret_cast<float *>(base + L.g1);

    ValidateArgs va;
    std::memset(&va, 0, sizeof(va));
    va.s[0] = input_scale;
    va.recip[0] = g;
    va.E = E;
    va.narrays = 1;
    va.hdr = hdr;
    NV_CUDA(launch_validate(va, st), "launching the scale check");
    DevHeader h;
    int rc = read_header(hdr, st, &h);
    if (rc) return rc;
    if (h.status) return header_status(h, nullptr);
    if (T == 0) {
        NV_CUDA(cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E + 1), st), "zeroing offsets");
        NV_CUDA(cudaStreamSynchronize(st), "synchronising the stream");
        return NVFP4_OK;
    }
    const int R = T * k;
    RouteArgs ra;
    std::memset(&ra, 0, sizeof(ra));
    ra.ids = topk_ids;
    ra.R = R;
    ra.k = k;
    ra.E = E;
    ra.nchunks = L.nchunks;
    ra.chunk_hist = reinterpret_cast<int *>(base + L.chunk_hist);
    ra.counts = reinterpret_cast<int *>(base + L.counts);
    ra.offsets = reinterpret_cast<int *>(base + L.offsets);
    ra.pad_off = reinterpret_cast<int *>(base + L.pad_off);
    ra.tile_expert = nullptr;
    ra.row_of = reinterpret_cast<int *>(base + L.row_of);
    ra.perm = perm;
    ra.row_src = nullptr;
    ra.offsets_out = expert_offsets;
    ra.pad_rows = 128;
    ra.padded = 0;
    ra.hdr = hdr;
    NV_CUDA(launch_route(ra, st), "launching the token reorder");
    const int kc = (H + 63) / 64;
    if (sf_layout == NVFP4_SF_SWIZZLED)
        NV_CUDA(cudaMemsetAsync(sf_out, 0, (size_t)((R + 127) / 128) * kc * 512, st), "zeroing scale padding");
    QuantArgs qa;
    std::memset(&qa, 0, sizeof(qa));
    qa.x = x;
    qa.ids = topk_ids;
    qa.row_of = ra.row_of;
    qa.g = g;
    qa.T = T;
    qa.H = H;
    qa.k = k;
    qa.q = q_out;
    qa.sf = sf_out;
    qa.sf_swizzled = sf_layout == NVFP4_SF_SWIZZLED;
    qa.sf_kc = kc;
    qa.sf_ue8m0 = sf_ue8m0;
    qa.hdr = hdr;
    NV_CUDA(launch_quant_experts(qa, st), "launching the quantiser");
    rc = read_header(hdr, st, &h);
    if (rc) return rc;
    return header_status(h, nullptr);
}

// The prepared buffer ends with a 256-byte slot whose first word names the
// block-scale format the scales were converted from; the forward checks it.
constexpr uint32_t kPrepTagE4M3 = 0xE4E4E4E4u, kPrepTagUE8M0 = 0x5E5E5E5Eu;
// UE8M0 weight-row factors after both scale layouts: [E, 2I] (w13) then [E, H] (w2).
static size_t prep_factor_offset(int E, int H, int I)
{
    return up256(prepared_w13_bytes(E, H, I)) + up256(prepared_w2_bytes(E, H, I));
}
static size_t prep_tag_offset(int E, int H, int I)
{
    return prep_factor_offset(E, H, I) + up256(sizeof(float) * (size_t)E * (2 * (size_t)I + H));
}

size_t nvfp4_prepared_weights_size(int E, int H, int I)
{
    if (E < 1 || H <= 0 || I <= 0) return 0;
    return prep_tag_offset(E, H, I) + 256;
}

static int check_weights(const nvfp4_moe_weights *w)
{
    if (!w) return fail(NVFP4_ERR_INVALID_ARG, "weights struct is null");
    if (!w->w13_q || !w->w13_sf || !w->w13_scale2 || !w->w13_input_scale || !w->w2_q || !w->w2_sf ||
        !w->w2_scale2 || !w->w2_input_scale)
        return fail(NVFP4_ERR_INVALID_ARG, "a weight or scale pointer is null");
    if (!aligned(w->w13_q, 16) || !aligned(w->w2_q, 16) || !aligned(w->w13_sf, 4) || !aligned(w->w2_sf, 4))
        return fail(NVFP4_ERR_INVALID_ARG, "weight codes must be 16-byte aligned, scales 4-byte aligned");
    return NVFP4_OK;
}

int nvfp4_prepare_weights(const nvfp4_moe_weights *w, void *prepared, size_t prepared_bytes, nvfp4_stream_t stream)
{
    return nvfp4_prepare_weights_format(w, prepared, prepared_bytes, NVFP4_SF_E4M3, stream);
}

int nvfp4_prepare_weights_format(const nvfp4_moe_weights *w, void *prepared, size_t prepared_bytes, int format,
                                 nvfp4_stream_t stream)
{
    if (format != NVFP4_SF_E4M3 && format != NVFP4_SF_UE8M0)
        return fail(NVFP4_ERR_INVALID_ARG, "prepare: unknown block-scale format %d", format);
    const int ue = format == NVFP4_SF_UE8M0;
    int rc = check_weights(w);
    if (rc) return rc;
    rc = check_layer_shape(w->E, w->H, w->I, 1);
    if (rc) return rc;
    if (!prepared || !aligned(prepared, 256)) return fail(NVFP4_ERR_INVALID_ARG, "prepared buffer null or misaligned");
    const size_t need = nvfp4_prepared_weights_size(w->E, w->H, w->I);
    if (prepared_bytes < need)
        return fail(NVFP4_ERR_WORKSPACE_TOO_SMALL, "prepared buffer %zu < %zu", prepared_bytes, need);
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t *base = static_cast<uint8_t *>(prepared);
    float *factors = reinterpret_cast<float *>(base + prep_factor_offset(w->E, w->H, w->I));
    PrepArgs a13 = {w->w13_sf, base, w->E, 2 * w->I, w->H, 4 * ((w->H + 255) / 256), w->I, ue, factors};
    NV_CUDA(launch_prep_sf(a13, st), "launching the w13 scale conversion");
    PrepArgs a2 = {w->w2_sf, base + up256(prepared_w13_bytes(w->E, w->H, w->I)), w->E, w->H, w->I,
                   4 * ((w->I + 255) / 256), 0, ue, factors + (size_t)w->E * 2 * w->I};
    NV_CUDA(launch_prep_sf(a2, st), "launching the w2 scale conversion");
    NV_CUDA(cudaMemsetAsync(base + prep_tag_offset(w->E, w->H, w->I), ue ? 0x5E : 0xE4, 4, st),
            "writing the format word");
    return NVFP4_OK;
}

size_t nvfp4_moe_workspace_size(int T, int H, int I, int E, int k)
{
    if (T < 0 || H <= 0 || I <= 0 || E < 1 || k < 1 || (long long)T * k > INT_MAX) return 0;
    return make_layout(T, H, I, E, k).end;
}

size_t nvfp4_moe_host_workspace_size(int T, int H, int I, int E, int k)
{
    if (T < 0 || H <= 0 || I <= 0 || E < 1 || k < 1 || (long long)T * k > INT_MAX) return 0;
    return make_layout(T, H, I, E, k).host_end;
}

static int forward_impl(const nvfp4_moe_weights *w, const void *prepared, const uint16_t *x, int T,
                        const int32_t *ids, const float *topk_w, int k, float *out, void *ws, size_t ws_bytes,
                        unsigned flags, cudaStream_t st, void *const *events = nullptr)
{
    auto mark = [&](int i) -> cudaError_t {
        return events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) : cudaSuccess;
    };
    int rc = check_weights(w);
    if (rc) return rc;
    rc = check_layer_shape(w->E, w->H, w->I, k);
    if (rc) return rc;
    const int E = w->E, H = w->H, I = w->I;
    if (T < 0) return fail(NVFP4_ERR_INVALID_ARG, "T=%d < 0", T);
    if ((long long)T * k >= (1ll << 31) / 2) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "T*k too large");
    if (!quant_offsets_fit(make_layout(T, H, I, E, k).rows_cap, H))
        return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "T*k too large for 32-bit scale offsets at H=%d", H);
    if (!prepared || !ws || (T > 0 && (!x || !ids || !topk_w || !out)))
        return fail(NVFP4_ERR_INVALID_ARG, "forward: null pointer");
    if (!aligned(ws, 256) || !aligned(prepared, 256) || (T > 0 && (!aligned(x, 16) || !aligned(out, 16))))
        return fail(NVFP4_ERR_INVALID_ARG, "forward: misaligned pointer (x, out 16 B; ws, prepared 256 B)");
    const WsLayout L = make_layout(T, H, I, E, k);
    if (ws_bytes < L.end) return fail(NVFP4_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu", ws_bytes, L.end);
    const bool keep_h = (flags & NVFP4_DEBUG_KEEP_H) != 0;
    const bool ue = (flags & NVFP4_UE8M0_SCALES) != 0;
    if ((flags & NVFP4_W13_ONE_SM) && (flags & NVFP4_W13_TWO_SM))
        return fail(NVFP4_ERR_INVALID_ARG, "NVFP4_W13_ONE_SM and NVFP4_W13_TWO_SM together");
    // w13 on CTA pairs when experts hold many rows on average: the rows are
    // then padded to 256 per expert, which costs a 128-row tile of padding on
    // about half the experts; with few rows per expert that costs more than
    // the pairs save
    const bool pairs = (flags & NVFP4_W13_TWO_SM) ||
                       (!(flags & NVFP4_W13_ONE_SM) && (long long)T * k >= kPairRowsPerExpert * (long long)E);
    if (keep_h && ws_bytes < L.host_end + (size_t)L.rows_cap * I * sizeof(float))
        return fail(NVFP4_ERR_WORKSPACE_TOO_SMALL, "NVFP4_DEBUG_KEEP_H needs the host workspace size + rows_cap*I*4");
    if (T == 0) return NVFP4_OK;

    uint8_t *base = static_cast<uint8_t *>(ws);
    DevHeader *hdr = reinterpret_cast<DevHeader *>(base + L.hdr);
    float *g = reinterpret_cast<float *>(base + L.g1);  // g1 | g2 | gw13 | gw2
    float *alpha1 = reinterpret_cast<float *>(base + L.alpha1);
    float *alpha2 = reinterpret_cast<float *>(base + L.alpha2);

    ValidateArgs va;
    std::memset(&va, 0, sizeof(va));
    va.s[0] = w->w13_input_scale;
    va.s[1] = w->w2_input_scale;
    va.s[2] = w->w13_scale2;
    va.s[3] = w->w2_scale2;
    va.written[0] = w->w13_input_written;
    va.written[1] = w->w2_input_written;
    for (int i = 0; i < 4; ++i) va.recip[i] = g + (size_t)i * E;
    va.E = E;
    va.narrays = 4;
    va.alpha1 = alpha1;
    va.alpha2 = alpha2;
    va.prep_tag = reinterpret_cast<const uint32_t *>(static_cast<const uint8_t *>(prepared) +
                                                     prep_tag_offset(E, H, I));
    va.prep_tag_want = ue ? kPrepTagUE8M0 : kPrepTagE4M3;
    va.hdr = hdr;
    const int R = T * k;
    RouteArgs ra;
    std::memset(&ra, 0, sizeof(ra));
    ra.ids = ids;
    ra.R = R;
    ra.k = k;
    ra.E = E;
    ra.nchunks = L.nchunks;
    ra.chunk_hist = reinterpret_cast<int *>(base + L.chunk_hist);
    ra.counts = reinterpret_cast<int *>(base + L.counts);
    ra.offsets = reinterpret_cast<int *>(base + L.offsets);
    ra.pad_off = reinterpret_cast<int *>(base + L.pad_off);
    ra.tile_expert = reinterpret_cast<int *>(base + L.tile_expert);
    ra.row_of = reinterpret_cast<int *>(base + L.row_of);
    ra.perm = reinterpret_cast<int *>(base + L.perm);
    ra.row_src = reinterpret_cast<int *>(base + L.row_src);
    int *row_max = reinterpret_cast<int *>(base + L.row_max);  // UE8M0: a1 rows, then a2 rows
    ra.row_max = ue ? row_max : nullptr;
    ra.rows_cap = L.rows_cap;
    ra.pad_rows = pairs ? 256 : 128;
    ra.live_mtiles = pairs ? reinterpret_cast<int *>(base + L.live_mtiles) : nullptr;
    ra.padded = 1;
    ra.hdr = hdr;

    // The w13 GEMM's small-batch plan when its waves of 64-column tiles (over
    // at most min(R, E) busy experts) take less time than the wide plan's
    // waves; a narrow tile's K loop takes about 0.55 of a wide one's.  It
    // quantises A itself, routing its own tile, when every CTA gets one tile
    // (busy experts x 64-column tiles within the SM count; at most
    // kSmallPlanRows <= 128 rows: one m-tile per busy expert), K fits its
    // persistent A buffer, and the routing runs as one kernel (not in timed
    // calls, which separate the scale check from the routing).
    const long long sms = sm_count();
    bool small_w13, a_inline;
    {
        const long long busy = std::min<long long>((long long)R, E);
        const long long small_waves = (busy * ((I + 63) / 64) + sms - 1) / sms;
        const long long wide_waves = (busy * ((I + 127) / 128) + sms - 1) / sms;
        small_w13 = !pairs && !ue && !(flags & NVFP4_W13_ONE_SM) && (long long)R <= kSmallPlanRows &&
                    100 * small_waves < 182 * wide_waves;
        a_inline = small_w13 && !events && busy * ((I + 63) / 64) <= sms && (long long)H <= kInlineQuantMaxK;
    }
    // otherwise, with the wide tiles on single CTAs and up to kEarlyRows
    // routed rows, w13 routes its tiles itself and starts its weight loads
    // before its dependency wait
    const bool early_w13 = !small_w13 && !pairs && !ue && !events && (long long)R <= kEarlyRows && E <= 1024;
    // and with the self-routed w13, w2's small-batch plan does the same (its
    // A loads after the wait).  Measured: 0.3-0.7 us less per 1-token call;
    // with the quantiser's path (2 to 8 tokens) up to 0.7 us more, so not there.
    const bool early_w2 = a_inline && (long long)R <= kSmallPlanRowsW2 && (long long)R <= kEarlyRows;
    // the a1 quantiser forms its row map from the ids and runs beside the routing
    const bool self_quant = !a_inline && !pairs && !ue && !events && (long long)R <= kEarlyRows && E <= 1024;
    // (the kernels above read the call's inputs before their dependency waits)
    ra.trigger_after_wait = (a_inline || early_w13 || early_w2 || self_quant) ? 1 : 0;
    // The routing returns at once when the check has failed, so it may be
    // queued before the host reads the status.  Timed calls keep the two
    // launches apart so that each has its own interval.
    NV_CUDA(mark(0), "recording an event");
    if (events) {
        NV_CUDA(launch_validate(va, st), "launching the scale check");
        NV_CUDA(mark(1), "recording an event");
        NV_CUDA(launch_route(ra, st), "launching the token reorder");
    } else {
        NV_CUDA(launch_validate_route(va, ra, st), "launching the scale check and the token reorder");
    }
    NV_CUDA(mark(2), "recording an event");
    if (!(flags & NVFP4_SCALES_PREVALIDATED)) {
        DevHeader h;
        rc = read_header(hdr, st, &h);
        if (rc) return rc;
        if (h.status) return header_status(h, nullptr);
    }

    if (!a_inline) {
        QuantArgs qa;
        std::memset(&qa, 0, sizeof(qa));
        qa.x = x;
        qa.ids = ids;
        qa.row_of = ra.row_of;
        qa.g = g;
        qa.T = T;
        qa.H = H;
        qa.k = k;
        qa.q = base + L.a1q;
        qa.sf = base + L.sf1;
        qa.sf_swizzled = 1;
        qa.sf_kc = L.kc1;
        qa.sf_ue8m0 = ue ? 1 : 0;  // UE8M0 bytes, carried to the tensor cores per row by the GEMM
        qa.row_max = ue ? row_max : nullptr;
        qa.hdr = hdr;
        qa.self_route = self_quant ? 1 : 0;
        qa.in_scale = w->w13_input_scale;
        qa.E = E;
        NV_CUDA(launch_quant_experts(qa, st), "launching the a1 quantiser");
    }
    NV_CUDA(mark(3), "recording an event");

    const uint8_t *pw = static_cast<const uint8_t *>(prepared);
    GemmArgs ga;
    std::memset(&ga, 0, sizeof(ga));
    ga.a_q = base + L.a1q;
    ga.b_q = w->w13_q;
    ga.a_sf = base + L.sf1;
    ga.b_sf = pw;
    ga.rows_cap = L.rows_cap;
    ga.K = H;
    ga.N = 2 * I;
    ga.E = E;
    ga.a_kc = L.kc1;
    ga.b_kc = L.kc1;
    ga.gate_up_I = I;
    ga.tile_expert = ra.tile_expert;
    ga.pad_off = ra.pad_off;
    ga.counts = ra.counts;
    ga.alpha = alpha1;
    ga.g2 = g + E;
    ga.a2q = base + L.a2q;
    ga.sf2 = base + L.sf2;
    ga.I = I;
    ga.kc2 = L.kc2;
    ga.h_dump = keep_h ? reinterpret_cast<float *>(base + L.host_end) : nullptr;
    ga.ue8m0 = ue ? 1 : 0;
    const float *factors = reinterpret_cast<const float *>(pw + prep_factor_offset(E, H, I));
    if (ue) {
        ga.a_row_max = row_max;
        ga.out_row_max = row_max + L.rows_cap;
        ga.b_row_factor = factors;
    }
    ga.zero_out = out;  // cleared by the w13 kernel for the w2 kernel's reductions
    ga.zero_floats = (long long)T * H;
    ga.k = k;
    ga.H = H;
    ga.hdr = hdr;
    ga.mtiles_cap = L.mtiles_cap;
    ga.pairs = pairs ? 1 : 0;
    ga.small = small_w13 ? 1 : 0;
    ga.a_inline = a_inline ? 1 : 0;
    ga.early = early_w13 ? 1 : 0;
    ga.x = x;
    ga.ids = ids;
    ga.R = R;
    ga.in_scale1 = w->w13_input_scale;
    ga.in_scale2 = w->w2_input_scale;
    ga.w13_scale2 = w->w13_scale2;
    NV_CUDA(launch_gemm_w13(ga, st), "launching the w13 GEMM");
    NV_CUDA(mark(4), "recording an event");

    GemmArgs gb = ga;
    gb.a_q = base + L.a2q;
    gb.b_q = w->w2_q;
    gb.a_sf = base + L.sf2;
    gb.b_sf = pw + up256(prepared_w13_bytes(E, H, I));
    gb.K = I;
    gb.N = H;
    gb.a_kc = L.kc2;
    gb.b_kc = L.kc2;
    gb.gate_up_I = 0;
    gb.alpha = alpha2;
    gb.h_dump = nullptr;
    gb.row_src = ra.row_src;
    gb.a_inline = 0;
    gb.topk_w = topk_w;
    gb.out = out;
    gb.pairs = 0;
    gb.small = !ue && (long long)T * k <= kSmallPlanRowsW2;
    gb.early = early_w2 ? 1 : 0;
    gb.live_mtiles = ra.live_mtiles;  // with 256-row padding, the m-tiles that hold rows
    if (ue) {
        gb.a_row_max = row_max + L.rows_cap;
        gb.out_row_max = nullptr;
        gb.b_row_factor = factors + (size_t)E * 2 * I;
    }
    NV_CUDA(launch_gemm_w2(gb, st), "launching the w2 GEMM");
    NV_CUDA(mark(5), "recording an event");

    if (flags & NVFP4_SYNC_CHECK) {
        DevHeader h;
        rc = read_header(hdr, st, &h);
        if (rc) return rc;
        return header_status(h, nullptr);
    }
    return NVFP4_OK;
}

int nvfp4_moe_forward(const nvfp4_moe_weights *w, const void *prepared, const uint16_t *x, int T,
                      const int32_t *topk_ids, const float *topk_weights, int k, float *out, void *ws,
                      size_t ws_bytes, unsigned flags, nvfp4_stream_t stream)
{
    return forward_impl(w, prepared, x, T, topk_ids, topk_weights, k, out, ws, ws_bytes, flags,
                        (cudaStream_t)stream);
}

int nvfp4_moe_forward_profiled(const nvfp4_moe_weights *w, const void *prepared, const uint16_t *x, int T,
                               const int32_t *topk_ids, const float *topk_weights, int k, float *out, void *ws,
                               size_t ws_bytes, unsigned flags, nvfp4_stream_t stream, void *const *events)
{
    if (!events) return fail(NVFP4_ERR_INVALID_ARG, "events is null");
    for (int i = 0; i < 6; ++i)
        if (!events[i]) return fail(NVFP4_ERR_INVALID_ARG, "event %d is null", i);
    return forward_impl(w, prepared, x, T, topk_ids, topk_weights, k, out, ws, ws_bytes, flags,
                        (cudaStream_t)stream, events);
}

// Token chunks of the pipelined host entry point.  Tokens are independent, so
// the layer runs chunk by chunk while the next chunk's inputs are copied in
// and the previous chunk's output is copied out.  Small first and last chunks
// shorten the copy-in head and the copy-out tail that nothing overlaps; the
// middle chunks are large enough to keep the GEMMs efficient.
static std::vector<std::pair<int, int>> host_chunks(int T)
{
    std::vector<std::pair<int, int>> c;
    constexpr int kEdge = 2048, kMid = 4096;
    if (T < 2 * kEdge) {
        c.push_back({0, T});
        return c;
    }
    const int mid = T - 2 * kEdge;
    int nmid = mid == 0 ? 0 : (mid + kMid - 1) / kMid;
    if (nmid > kMaxHostChunks - 2) nmid = kMaxHostChunks - 2;
    c.push_back({0, kEdge});
    int t0 = kEdge;
    for (int i = 0; i < nmid; ++i) {
        const int n = (mid - (t0 - kEdge) + (nmid - i) - 1) / (nmid - i);
        c.push_back({t0, n});
        t0 += n;
    }
    c.push_back({t0, kEdge});
    return c;
}

namespace {
// Copy streams and events of the host entry point, one set per device,
// created on first use.  A call holds the device's mutex from its first
// enqueue to its final synchronisation, so sets are never shared by two calls.
struct HostPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, in_done[kMaxHostChunks], fwd_done[kMaxHostChunks], out_done[kMaxHostChunks];
};
HostPipe g_pipes[64];
}  // namespace

int nvfp4_moe_forward_host(const nvfp4_moe_weights *w, const void *prepared, const uint16_t *x_host, int T,
                           const int32_t *topk_ids_host, const float *topk_weights_host, int k, float *out_host,
                           void *ws, size_t ws_bytes, unsigned flags, nvfp4_stream_t stream)
{
    int rc = check_weights(w);
    if (rc) return rc;
    rc = check_layer_shape(w->E, w->H, w->I, k);
    if (rc) return rc;
    if (T < 0 || !ws || (T > 0 && (!x_host || !topk_ids_host || !topk_weights_host || !out_host)))
        return fail(NVFP4_ERR_INVALID_ARG, "forward_host: bad arguments");
    const WsLayout L = make_layout(T, w->H, w->I, w->E, k);
    if (ws_bytes < L.host_end)
        return fail(NVFP4_ERR_WORKSPACE_TOO_SMALL, "host workspace %zu < %zu", ws_bytes, L.host_end);
    if (T == 0) return NVFP4_OK;
    int dev = 0;
    NV_CUDA(cudaGetDevice(&dev), "querying the device");
    if (dev < 0 || dev >= 64) return fail(NVFP4_ERR_CUDA, "device %d out of range", dev);
    HostPipe &P = g_pipes[dev];
    std::lock_guard<std::mutex> lock(P.mu);
    if (!P.ready) {
        NV_CUDA(cudaStreamCreateWithFlags(&P.in, cudaStreamNonBlocking), "creating a copy stream");
        NV_CUDA(cudaStreamCreateWithFlags(&P.out, cudaStreamNonBlocking), "creating a copy stream");
        NV_CUDA(cudaEventCreateWithFlags(&P.start, cudaEventDisableTiming), "creating an event");
        for (int i = 0; i < kMaxHostChunks; ++i) {
            NV_CUDA(cudaEventCreateWithFlags(&P.in_done[i], cudaEventDisableTiming), "creating an event");
            NV_CUDA(cudaEventCreateWithFlags(&P.fwd_done[i], cudaEventDisableTiming), "creating an event");
            NV_CUDA(cudaEventCreateWithFlags(&P.out_done[i], cudaEventDisableTiming), "creating an event");
        }
        P.ready = true;
    }
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t *base = static_cast<uint8_t *>(ws);
    uint16_t *x = reinterpret_cast<uint16_t *>(base + L.x_stage);
    int32_t *ids = reinterpret_cast<int32_t *>(base + L.ids_stage);
    float *tw = reinterpret_cast<float *>(base + L.w_stage);
    float *out = reinterpret_cast<float *>(base + L.out_stage);
    DevHeader *status = reinterpret_cast<DevHeader *>(base + L.status_stage);
    const size_t H = (size_t)w->H;
    const std::vector<std::pair<int, int>> chunks = host_chunks(T);
    const int n = (int)chunks.size();

    // Everything already on the caller's stream (earlier users of this
    // workspace) completes before the copy streams touch it.
    NV_CUDA(cudaEventRecord(P.start, st), "recording an event");
    NV_CUDA(cudaStreamWaitEvent(P.in, P.start, 0), "ordering the copy stream");
    NV_CUDA(cudaStreamWaitEvent(P.out, P.start, 0), "ordering the copy stream");
    for (int c = 0; c < n; ++c) {
        const size_t t0 = (size_t)chunks[c].first, tc = (size_t)chunks[c].second;
        NV_CUDA(cudaMemcpyAsync(x + t0 * H, x_host + t0 * H, sizeof(uint16_t) * tc * H, cudaMemcpyHostToDevice, P.in),
                "copying x");
        NV_CUDA(cudaMemcpyAsync(ids + t0 * k, topk_ids_host + t0 * k, sizeof(int32_t) * tc * k,
                                cudaMemcpyHostToDevice, P.in),
                "copying ids");
        NV_CUDA(cudaMemcpyAsync(tw + t0 * k, topk_weights_host + t0 * k, sizeof(float) * tc * k,
                                cudaMemcpyHostToDevice, P.in),
                "copying weights");
        NV_CUDA(cudaEventRecord(P.in_done[c], P.in), "recording an event");
    }
    int first_rc = NVFP4_OK;
    for (int c = 0; c < n; ++c) {
        const size_t t0 = (size_t)chunks[c].first;
        const int tc = chunks[c].second;
        NV_CUDA(cudaStreamWaitEvent(st, P.in_done[c], 0), "ordering the compute stream");
        // The first chunk checks the scales as the caller asked (with a host
        // synchronisation unless they were pre-validated); the device keeps
        // checking them in every chunk, and each chunk's status is saved.
        const unsigned cf = (flags & ~(NVFP4_DEBUG_KEEP_H | NVFP4_SYNC_CHECK)) |
                            (c > 0 ? (unsigned)NVFP4_SCALES_PREVALIDATED : 0u);
        rc = forward_impl(w, prepared, x + t0 * H, tc, ids + t0 * k, tw + t0 * k, k, out + t0 * H, ws, ws_bytes,
                          cf, st);
        if (rc) {
            first_rc = rc;
            break;
        }
        NV_CUDA(cudaMemcpyAsync(status + c, base + L.hdr, sizeof(DevHeader), cudaMemcpyDeviceToDevice, st),
                "saving the chunk status");
        NV_CUDA(cudaEventRecord(P.fwd_done[c], st), "recording an event");
        NV_CUDA(cudaStreamWaitEvent(P.out, P.fwd_done[c], 0), "ordering the copy stream");
        NV_CUDA(cudaMemcpyAsync(out_host + t0 * H, out + t0 * H, sizeof(float) * (size_t)tc * H,
                                cudaMemcpyDeviceToHost, P.out),
                "copying out");
        NV_CUDA(cudaEventRecord(P.out_done[c], P.out), "recording an event");
    }
    // Nothing of this call is left in flight when it returns: the caller may
    // reuse its host buffers at once, also after an error.
    NV_CUDA(cudaStreamSynchronize(P.in), "synchronising the copy stream");
    NV_CUDA(cudaStreamSynchronize(P.out), "synchronising the copy stream");
    if (first_rc) {
        NV_CUDA(cudaStreamSynchronize(st), "synchronising the stream");
        return first_rc;
    }
    DevHeader h[kMaxHostChunks];
    NV_CUDA(cudaMemcpyAsync(h, status, sizeof(DevHeader) * n, cudaMemcpyDeviceToHost, st), "reading the status");
    NV_CUDA(cudaStreamSynchronize(st), "synchronising the stream");
    for (int c = 0; c < n; ++c) {
        rc = header_status(h[c], nullptr);
        if (rc) return rc;
    }
    return NVFP4_OK;
}

int nvfp4_moe_status(const void *ws, nvfp4_stream_t stream, int *first_bad_host)
{
    if (!ws) return fail(NVFP4_ERR_INVALID_ARG, "ws is null");
    DevHeader h;
    int rc = read_header(ws, (cudaStream_t)stream, &h);
    if (rc) return rc;
    return header_status(h, first_bad_host);
}

int nvfp4_moe_intermediates_of(void *ws, int T, int H, int I, int E, int k, nvfp4_moe_intermediates *o)
{
    if (!ws || !o) return fail(NVFP4_ERR_INVALID_ARG, "null argument");
    const WsLayout L = make_layout(T, H, I, E, k);
    uint8_t *b = static_cast<uint8_t *>(ws);
    o->rows_cap = L.rows_cap;
    o->a1q = b + L.a1q;
    o->sf1 = b + L.sf1;
    o->a2q = b + L.a2q;
    o->sf2 = b + L.sf2;
    o->row_of = reinterpret_cast<int32_t *>(b + L.row_of);
    o->offsets = reinterpret_cast<int32_t *>(b + L.offsets);
    o->pad_offsets = reinterpret_cast<int32_t *>(b + L.pad_off);
    o->h = reinterpret_cast<float *>(b + L.host_end);
    return NVFP4_OK;
}

// ---------------------------------------------------------------- W4A16
static int check_weights_w16(const nvfp4_moe_weights *w)
{
    if (!w) return fail(NVFP4_ERR_INVALID_ARG, "weights struct is null");
    if (!w->w13_q || !w->w13_sf || !w->w13_scale2 || !w->w2_q || !w->w2_sf || !w->w2_scale2)
        return fail(NVFP4_ERR_INVALID_ARG, "a weight or weight-scale pointer is null");
    if (!aligned(w->w13_q, 16) || !aligned(w->w2_q, 16) || !aligned(w->w13_sf, 4) || !aligned(w->w2_sf, 4))
        return fail(NVFP4_ERR_INVALID_ARG, "weight codes must be 16-byte aligned, scales 4-byte aligned");
    return NVFP4_OK;
}

static size_t w16_w13_sf_bytes(int E, int H, int I) { return (size_t)E * 2 * I * (H / 16); }

size_t nvfp4_w4a16_prepared_size(int E, int H, int I)
{
    if (E < 1 || H <= 0 || I <= 0 || H % 64 || I % 64) return 0;
    return up256(w16_w13_sf_bytes(E, H, I)) + up256((size_t)E * H * (I / 16));
}

int nvfp4_prepare_weights_w4a16(const nvfp4_moe_weights *w, void *prepared, size_t prepared_bytes,
                                nvfp4_stream_t stream)
{
    int rc = check_weights_w16(w);
    if (rc) return rc;
    rc = check_layer_shape(w->E, w->H, w->I, 1);
    if (rc) return rc;
    if (!prepared || !aligned(prepared, 256)) return fail(NVFP4_ERR_INVALID_ARG, "prepared: null or not 256-byte aligned");
    if (prepared_bytes < nvfp4_w4a16_prepared_size(w->E, w->H, w->I))
        return fail(NVFP4_ERR_WORKSPACE_TOO_SMALL, "prepared buffer too small");
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t *base = static_cast<uint8_t *>(prepared);
    NV_CUDA(launch_prep_sf_w16(w->w13_sf, base, w->E, 2 * w->I, w->H, st), "launching the w13 scale layout");
    NV_CUDA(launch_prep_sf_w16(w->w2_sf, base + up256(w16_w13_sf_bytes(w->E, w->H, w->I)), w->E, w->H, w->I, st),
            "launching the w2 scale layout");
    return NVFP4_OK;
}

// W4A16 workspace: the routing regions of the W4A4 layout, then A (gathered
// BF16 rows, [rows_cap, H]) and h ([rows_cap, I] BF16) in place of the W4A4
// activation buffers.
struct W16Layout {
    size_t a16, h16, end;
};
static W16Layout make_w16_layout(const WsLayout &L, int H, int I)
{
    W16Layout w;
    w.a16 = L.a1q;
    w.h16 = w.a16 + up256((size_t)L.rows_cap * H * 2);
    w.end = w.h16 + up256((size_t)L.rows_cap * I * 2);
    return w;
}

size_t nvfp4_moe_w4a16_workspace_size(int T, int H, int I, int E, int k)
{
    if (T < 0 || H <= 0 || I <= 0 || E < 1 || k < 1) return 0;
    const WsLayout L = make_layout(T, H, I, E, k);
    return make_w16_layout(L, H, I).end;
}

int nvfp4_moe_forward_w4a16(const nvfp4_moe_weights *w, const void *prepared, const uint16_t *x, int T,
                            const int32_t *topk_ids, const float *topk_weights, int k, float *out, void *ws,
                            size_t ws_bytes, unsigned flags, nvfp4_stream_t stream)
{
    int rc = check_weights_w16(w);
    if (rc) return rc;
    rc = check_layer_shape(w->E, w->H, w->I, k);
    if (rc) return rc;
    const int E = w->E, H = w->H, I = w->I;
    if (T < 0) return fail(NVFP4_ERR_INVALID_ARG, "T=%d < 0", T);
    if (flags & NVFP4_UE8M0_SCALES)
        return fail(NVFP4_ERR_INVALID_ARG, "w4a16 forward: UE8M0 weight scales are not supported");
    if ((long long)T * k >= (1ll << 31) / 2) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "T*k too large");
    if (!prepared || !ws || (T > 0 && (!x || !topk_ids || !topk_weights || !out)))
        return fail(NVFP4_ERR_INVALID_ARG, "w4a16 forward: null pointer");
    if (!aligned(ws, 256) || !aligned(prepared, 256) || (T > 0 && (!aligned(x, 16) || !aligned(out, 16))))
        return fail(NVFP4_ERR_INVALID_ARG, "w4a16 forward: misaligned pointer (x, out 16 B; ws, prepared 256 B)");
    const WsLayout L = make_layout(T, H, I, E, k);
    const W16Layout W = make_w16_layout(L, H, I);
    if (ws_bytes < W.end) return fail(NVFP4_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu", ws_bytes, W.end);
    if (T == 0) return NVFP4_OK;
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t *base = static_cast<uint8_t *>(ws);
    DevHeader *hdr = reinterpret_cast<DevHeader *>(base + L.hdr);

    // only the weight_scale_2 slots are consumed (no activation scale)
    ValidateArgs va;
    std::memset(&va, 0, sizeof(va));
    va.s[0] = w->w13_scale2;
    va.s[1] = w->w2_scale2;
    va.E = E;
    va.narrays = 2;
    va.hdr = hdr;

    RouteArgs ra;
    std::memset(&ra, 0, sizeof(ra));
    ra.ids = topk_ids;
    ra.R = T * k;
    ra.k = k;
    ra.E = E;
    ra.nchunks = L.nchunks;
    ra.chunk_hist = reinterpret_cast<int *>(base + L.chunk_hist);
    ra.counts = reinterpret_cast<int *>(base + L.counts);
    ra.offsets = reinterpret_cast<int *>(base + L.offsets);
    ra.pad_off = reinterpret_cast<int *>(base + L.pad_off);
    ra.tile_expert = reinterpret_cast<int *>(base + L.tile_expert);
    ra.row_of = reinterpret_cast<int *>(base + L.row_of);
    ra.perm = reinterpret_cast<int *>(base + L.perm);
    ra.row_src = reinterpret_cast<int *>(base + L.row_src);
    ra.pad_rows = 128;
    ra.padded = 1;
    ra.hdr = hdr;
    NV_CUDA(launch_validate_route(va, ra, st), "launching the scale check and the token reorder");
    if (!(flags & NVFP4_SCALES_PREVALIDATED)) {
        DevHeader h;
        rc = read_header(hdr, st, &h);
        if (rc) return rc;
        if (h.status) return header_status(h, nullptr);
    }

    uint16_t *a16 = reinterpret_cast<uint16_t *>(base + W.a16);
    uint16_t *h16 = reinterpret_cast<uint16_t *>(base + W.h16);
    NV_CUDA(launch_gather_rows(x, H, k, ra.row_src, hdr, L.rows_cap, a16, out, (long long)T * H, st),
            "launching the row gather");

    const uint8_t *pw = static_cast<const uint8_t *>(prepared);
    W16Args wa;
    std::memset(&wa, 0, sizeof(wa));
    wa.a = a16;
    wa.b_q = w->w13_q;
    wa.b_sfp = pw;
    wa.rows_cap = L.rows_cap;
    wa.K = H;
    wa.N = 2 * I;
    wa.E = E;
    wa.gate_up_I = I;
    wa.tile_expert = ra.tile_expert;
    wa.pad_off = ra.pad_off;
    wa.counts = ra.counts;
    wa.row_src = ra.row_src;
    wa.scale2 = w->w13_scale2;
    wa.h = h16;
    wa.I = I;
    wa.k = k;
    wa.H = H;
    wa.hdr = hdr;
    wa.mtiles_cap = L.mtiles_cap;
    NV_CUDA(launch_w16_w13(wa, st), "launching the W4A16 w13 GEMM");

    W16Args wb = wa;
    wb.a = h16;
    wb.b_q = w->w2_q;
    wb.b_sfp = pw + up256(w16_w13_sf_bytes(E, H, I));
    wb.K = I;
    wb.N = H;
    wb.gate_up_I = 0;
    wb.scale2 = w->w2_scale2;
    wb.h = nullptr;
    wb.topk_w = topk_weights;
    wb.out = out;
    // column blocks per group: the largest divisor of H/128 whose output slice
    // (T rows x 128 G columns of FP32) stays within about 48 MB of L2
    const int nblk = H / 128;
    const long long per_blk = (long long)T * 128 * 4;
    wb.col_group = 1;
    for (int G = nblk; G >= 1; --G)
        if (nblk % G == 0 && (long long)G * per_blk <= (48ll << 20)) {
            wb.col_group = G;
            break;
        }
    NV_CUDA(launch_w16_w2(wb, st), "launching the W4A16 w2 GEMM");

    if (flags & NVFP4_SYNC_CHECK) {
        DevHeader h;
        rc = read_header(hdr, st, &h);
        if (rc) return rc;
        return header_status(h, nullptr);
    }
    return NVFP4_OK;
}

int nvfp4_moe_w4a16_intermediates_of(void *ws, int T, int H, int I, int E, int k, uint16_t **a16, uint16_t **h16)
{
    if (!ws || T < 0 || H <= 0 || I <= 0 || E < 1 || k < 1 || !a16 || !h16)
        return fail(NVFP4_ERR_INVALID_ARG, "w4a16 intermediates: bad arguments");
    const WsLayout L = make_layout(T, H, I, E, k);
    const W16Layout W = make_w16_layout(L, H, I);
    *a16 = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws) + W.a16);
    *h16 = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws) + W.h16);
    return NVFP4_OK;
}

int nvfp4_residual_rmsnorm(const uint16_t *x, const float *out, int T, int H, float eps, uint16_t *x_next,
                           nvfp4_stream_t stream)
{
    if (T < 0 || H <= 0 || (T > 0 && (!x || !out || !x_next)))
        return fail(NVFP4_ERR_INVALID_ARG, "rmsnorm: bad arguments");
    if (T == 0) return NVFP4_OK;
    NV_CUDA(launch_rmsnorm(x, out, T, H, eps, x_next, (cudaStream_t)stream), "launching residual + RMSNorm");
    return NVFP4_OK;
}

int nvfp4_router_topk(const void *logits, int logits_dtype, int T, int E, int k, int32_t *topk_ids,
                      float *topk_weights, nvfp4_stream_t stream)
{
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E)
        return fail(NVFP4_ERR_INVALID_ARG, "router_topk: need T >= 0, 1 <= E <= 1024, 1 <= k <= min(32, E)");
    if (logits_dtype != NVFP4_LOGITS_F32 && logits_dtype != NVFP4_LOGITS_BF16)
        return fail(NVFP4_ERR_INVALID_ARG, "router_topk: logits_dtype must be NVFP4_LOGITS_F32 or NVFP4_LOGITS_BF16");
    if (T == 0) return NVFP4_OK;
    if (!logits || !topk_ids || !topk_weights) return fail(NVFP4_ERR_INVALID_ARG, "router_topk: null pointer");
    if (!aligned(logits, logits_dtype == NVFP4_LOGITS_F32 ? 4 : 2) || !aligned(topk_ids, 4) || !aligned(topk_weights, 4))
        return fail(NVFP4_ERR_INVALID_ARG, "router_topk: misaligned pointer");
    NV_CUDA(launch_router_topk(logits, logits_dtype == NVFP4_LOGITS_BF16, T, E, k, topk_ids, topk_weights,
                               (cudaStream_t)stream),
            "launching the router");
    return NVFP4_OK;
}

size_t nvfp4_quantize_weights_workspace_size(int count) { return count > 0 ? up256(sizeof(unsigned) * count) : 0; }

int nvfp4_quantize_weights(const uint16_t *w, int count, int N, int K, uint8_t *q, uint8_t *sf, float *scale2,
                           void *ws, size_t ws_bytes, nvfp4_stream_t stream)
{
    return nvfp4_quantize_weights_format(w, count, N, K, 0, q, sf, scale2, ws, ws_bytes, stream);
}

int nvfp4_quantize_weights_format(const uint16_t *w, int count, int N, int K, int sf_format, uint8_t *q,
                                  uint8_t *sf, float *scale2, void *ws, size_t ws_bytes, nvfp4_stream_t stream)
{
    if (sf_format != 0 && sf_format != NVFP4_SF_UE8M0)
        return fail(NVFP4_ERR_INVALID_ARG, "quantize_weights: sf_format must be 0 (E4M3) or NVFP4_SF_UE8M0");
    if (count < 1 || count > 65535 || N < 1 || K < 16 || K % 16 != 0 || !w || !q || !sf || !scale2 || !ws)
        return fail(NVFP4_ERR_INVALID_ARG, "quantize_weights: bad arguments");
    if (!aligned(q, 8)) return fail(NVFP4_ERR_INVALID_ARG, "quantize_weights: q must be 8-byte aligned");
    if (ws_bytes < nvfp4_quantize_weights_workspace_size(count))
        return fail(NVFP4_ERR_WORKSPACE_TOO_SMALL, "quantize_weights: workspace too small");
    NV_CUDA(launch_quantize_weights(w, count, N, K, q, sf, scale2, static_cast<unsigned *>(ws),
                                    sf_format == NVFP4_SF_UE8M0, (cudaStream_t)stream),
            "launching the weight quantiser");
    return NVFP4_OK;
}

}  // extern "C"
