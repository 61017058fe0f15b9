// Memory-bound kernels of the NVFP4 MoE expert path (sm_103a):
//   scale validation, token reorder (histogram + scan + stable scatter),
//   the routed activation quantiser, the weight-scale layout conversion,
//   residual + RMSNorm, and the static weight quantiser.
//
// Page cited: "Gemma 4 NVFP4 MoE 空输出" (taking-lying-flat.github.io).
#include <climits>
#include <cfloat>

#include "internal.h"
#include "tc_common.cuh"

namespace nvfp4 {
namespace {

// ------------------------------------------------------------------ validate
// [page, ROOT CAUSE]: a per-expert scale slot left unwritten by the loader is
// reciprocated into an inf / NaN / garbage global scale.  Every slot must be
// written, finite, positive and normal, and so must its FP32 reciprocal.
// Run by one CTA of 256 threads; ends with the header written by thread 0
// and returns the status it wrote (every thread, after a block barrier).
__device__ __forceinline__ int validate_body(const ValidateArgs &a)
{
    __shared__ int s_bad, s_first, s_status;
    __shared__ float s_recip[4][1024];  // reciprocals for alpha (forward: 4 arrays, E <= 1024)
    // the format word is read first, so that its load overlaps the scale loads
    const uint32_t tag = threadIdx.x == 0 && a.prep_tag ? *a.prep_tag : a.prep_tag_want;
    if (threadIdx.x == 0) {
        s_bad = 0;
        s_first = INT_MAX;
    }
    __syncthreads();
    const int n = a.narrays * a.E;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int arr = i / a.E, e = i - arr * a.E;
        const float x = a.s[arr][e];
        bool ok = true;
        if (a.written[arr] && a.written[arr][e] == 0) ok = false;
        const float ax = fabsf(x);
        if (!(x > 0.0f) || !(ax <= FLT_MAX) || ax < FLT_MIN) ok = false;
        const float r = __frcp_rn(x);  // the reciprocal the format conversion takes
        const float ar = fabsf(r);
        if (!(ar <= FLT_MAX) || ar < FLT_MIN) ok = false;
        if (a.recip[arr]) a.recip[arr][e] = r;
        if (arr < 4 && e < 1024) s_recip[arr][e] = r;  // the forward's alpha needs E <= 1024, 4 arrays
        if (!ok) {
            atomicAdd(&s_bad, 1);
            atomicMin(&s_first, i);
        }
    }
    __syncthreads();
    // GEMM output scale 1/(g_a * g_w) per expert [page, §NVFP4 runtime-order
    // figure: the GEMM's scaling takes in both FP32 global scales].
    if (a.alpha1 && a.narrays == 4) {
        for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
            a.alpha1[e] = __frcp_rn(__fmul_rn(s_recip[0][e], s_recip[2][e]));
            a.alpha2[e] = __frcp_rn(__fmul_rn(s_recip[1][e], s_recip[3][e]));
        }
    }
    if (threadIdx.x == 0) {
        const bool tag_bad = tag != a.prep_tag_want;
        const int status = s_bad ? 2 : tag_bad ? 4 : 0;
        a.hdr->bad_count = s_bad;
        a.hdr->first_bad = s_first;
        a.hdr->status = status;
        a.hdr->error_flags = 0;
        a.hdr->num_mtiles = 0;
        a.hdr->done_count = 0u;
        s_status = status;
    }
    __syncthreads();
    return s_status;
}

__global__ void __launch_bounds__(256) validate_kernel(ValidateArgs a)
{
    pdl_trigger();
    pdl_wait();  // whatever ran before on the stream (a previous call may still read the header)
    validate_body(a);
}

// ------------------------------------------------------------------ routing
// [page, §矩阵融合 "MoE FFN"]: rows are reordered by expert so all experts'
// GEMMs run as one grouped GEMM.  Order inside an expert: ascending routed
// row f = t*k + j (stable), which makes the permutation unique.
//
// One cooperative launch (every CTA resident) over chunks of kRouteChunk
// routed rows, in two phases around a grid barrier:
//   1. per-chunk expert histograms (shared-memory atomics) -> chunk_hist;
//      an out-of-range id raises kErrBadExpertId.
//   2. every CTA reads all chunk histograms and forms, by warp scans, the
//      compact and 128-row-padded expert offsets (identical in every CTA); the
//      CTAs share out the m-tile -> expert map and the padding entries of
//      row_src; then each chunk is scattered: its warps own contiguous 256-row
//      slices, per-warp histograms give each warp's first rank per expert, and
//      equal experts inside a 32-row step are ranked with __match_any_sync.
// The barrier counter is the header's done_count, cleared by the scale check
// that precedes every routing launch; its wait is bounded.  A single CTA
// (up to kRouteChunk routed rows) needs no barrier, and then runs in the same
// kernel as the scale check (validate_route_kernel).
constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteSlice = kRouteChunk / kRouteWarps;  // rows per warp per chunk
constexpr int kRouteIdsPerLane = kRouteSlice / 32;
constexpr int kRouteMaxOwn = 8;  // chunks per CTA the shared-memory plan allows for

__device__ __forceinline__ void route_body(const RouteArgs &a)
{
    extern __shared__ int sh[];
    __shared__ int s_fail;
    const int E = a.E;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (a.hdr->status != 0) return;  // same value in every CTA (set by the scale check)
    if (tid == 0) s_fail = 0;

    // ---- phase 1: chunk histograms.  Each thread reads its ids in the
    // scatter's mapping (warp w: rows [256 w, 256 w + 256) of the chunk, lane l:
    // rows 32 i + l) all at once, and keeps those of its first chunk in
    // registers for the scatter.
    int *hist = sh;  // [E]
    int ids_first[kRouteIdsPerLane];
    for (int c = blockIdx.x; c < a.nchunks; c += gridDim.x) {
        for (int e = tid; e < E; e += kRouteThreads) hist[e] = 0;
        const int wf0 = c * kRouteChunk + warp * kRouteSlice;
        int idv[kRouteIdsPerLane];
#pragma unroll
        for (int i = 0; i < kRouteIdsPerLane; ++i) {
            const int f = wf0 + 32 * i + lane;
            idv[i] = f < a.R ? a.ids[f] : 0;
        }
        __syncthreads();
        bool bad = false;
#pragma unroll
        for (int i = 0; i < kRouteIdsPerLane; ++i) {
            if (wf0 + 32 * i + lane >= a.R) {
                idv[i] = -1;  // past the end: no row
            } else if (idv[i] < 0 || idv[i] >= E) {
                bad = true;
            } else {
                atomicAdd(&hist[idv[i]], 1);
            }
        }
        if (bad) atomicOr(&a.hdr->error_flags, kErrBadExpertId);
        if (c == (int)blockIdx.x) {
#pragma unroll
            for (int i = 0; i < kRouteIdsPerLane; ++i) ids_first[i] = idv[i];
        }
        __syncthreads();
        for (int e = tid; e < E; e += kRouteThreads) a.chunk_hist[(size_t)c * E + e] = hist[e];
        __syncthreads();
    }

    // ---- grid barrier (with one CTA, the block barrier below is enough: its
    // own global writes are visible to all its threads after it)
    if (tid == 0 && gridDim.x > 1) {
        __threadfence();
        atomicAdd(&a.hdr->done_count, 1u);
        const uint64_t t0 = global_timer_ns();
        for (;;) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(&a.hdr->done_count) : "memory");
            if (v >= gridDim.x) break;
            if (global_timer_ns() - t0 > 1000000000ull) {
                atomicOr(&a.hdr->error_flags, kErrTimeoutRoute);
                a.hdr->status = 5;
                s_fail = 1;
                break;
            }
        }
        __threadfence();
    }
    __syncthreads();
    if (s_fail) return;
    if (__ldcg(&a.hdr->error_flags) & kErrBadExpertId) {
        if (blockIdx.x == 0 && tid == 0) a.hdr->status = 3;  // nothing after this writes
        return;
    }
    // ---- phase 2: offsets (every CTA), this CTA's chunk prefixes
    const int own = (a.nchunks - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;  // chunks of this CTA
    int *cnt = sh;                    // [E]
    int *off = cnt + E;               // [E + 1]
    int *poff = off + E + 1;          // [E + 1]
    int *wbase = poff + E + 1;        // [kRouteWarps][E]
    int *cpre = wbase + kRouteWarps * E;  // [own][E]: chunk's first rank per expert
    int *psum = cpre + kRouteMaxOwn * E;  // [parts][E]
    int *loff = psum + (E > kRouteThreads ? E : kRouteThreads);  // [E + 1]: first live 128-row tile per expert
    // Per expert, the exclusive prefix over chunks.  With few experts the chunk
    // range is split into `parts` runs summed by different threads (one batch
    // of loads each), then the runs' sums are chained.
    const int parts = E >= kRouteThreads ? 1 : min(kRouteThreads / E, 16);
    const int csz = (a.nchunks + parts - 1) / parts;
    for (int t = tid; t < parts * E; t += kRouteThreads) {
        const int e = t % E, part = t / E;
        const int c_lo = part * csz, c_hi = min(a.nchunks, c_lo + csz);
        // this CTA's chunks are blockIdx.x + j * gridDim.x; the first at or after c_lo
        int j = c_lo <= (int)blockIdx.x ? 0 : (c_lo - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
        int next_own = (int)blockIdx.x + j * (int)gridDim.x;
        int run = 0;
        for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
            int v[16];
            const int n = min(16, c_hi - c0);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = i < n ? __ldcg(&a.chunk_hist[(size_t)(c0 + i) * E + e]) : 0;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (i < n && c0 + i == next_own) {
                    cpre[j * E + e] = run;  // prefix within this run, completed below
                    ++j;
                    next_own += gridDim.x;
                }
                run += v[i];
            }
        }
        psum[part * E + e] = run;
    }
    __syncthreads();
    for (int e = tid; e < E; e += kRouteThreads) {
        int before = 0, j = 0;
        for (int part = 0; part < parts; ++part) {
            const int c_hi = min(a.nchunks, (part + 1) * csz);
            for (; j < own && (int)blockIdx.x + j * (int)gridDim.x < c_hi; ++j) cpre[j * E + e] += before;
            before += psum[part * E + e];
        }
        cnt[e] = before;
        if (blockIdx.x == 0) a.counts[e] = before;
    }
    __syncthreads();
    // exclusive scans over experts by warp 0, 32 experts per step: compact,
    // padded to the pad_rows granularity (128, or 256 so that the 2-SM GEMM's
    // m-tile pairs belong to one expert), and the live 128-row tiles
    // (ceil(count / 128) per expert, the tiles holding rows)
    const int padm = (a.pad_rows == 256 ? 256 : 128) - 1;
    if (warp == 0) {
        int base_o = 0, base_p = 0, base_l = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int c = e < E ? cnt[e] : 0;
            const int cp = (c + padm) & ~padm;
            const int cl = (c + 127) >> 7;
            int io = c, ip = cp, il = cl;  // inclusive warp scans
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int to = __shfl_up_sync(0xffffffffu, io, o), tp = __shfl_up_sync(0xffffffffu, ip, o),
                          tl = __shfl_up_sync(0xffffffffu, il, o);
                if (lane >= o) {
                    io += to;
                    ip += tp;
                    il += tl;
                }
            }
            if (e < E) {
                off[e] = base_o + io - c;
                poff[e] = base_p + ip - cp;
                loff[e] = base_l + il - cl;
            }
            base_o += __shfl_sync(0xffffffffu, io, 31);
            base_p += __shfl_sync(0xffffffffu, ip, 31);
            base_l += __shfl_sync(0xffffffffu, il, 31);
        }
        if (lane == 0) {
            off[E] = base_o;
            poff[E] = base_p;
            loff[E] = base_l;
            if (blockIdx.x == 0) {
                a.hdr->num_mtiles = base_p >> 7;
                a.hdr->num_live_mtiles = base_l;
            }
        }
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int e = tid; e <= E; e += kRouteThreads) {
            a.offsets[e] = off[e];
            a.pad_off[e] = poff[e];
            if (a.offsets_out) a.offsets_out[e] = off[e];
        }
    }
    // m-tile -> expert map, shared out over the grid: binary search for the
    // last expert whose padded range starts at or before the tile
    if (a.tile_expert) {
        const int ntile = poff[E] >> 7;
        for (int mtile = blockIdx.x * kRouteThreads + tid; mtile < ntile; mtile += gridDim.x * kRouteThreads) {
            const int row = mtile << 7;
            int lo = 0, hi = E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (poff[mid] <= row)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            a.tile_expert[mtile] = lo;
        }
        // live tiles in order: live tile j of expert e is m-tile poff[e]/128 + (j - loff[e])
        if (a.live_mtiles) {
            const int nlive = loff[E];
            for (int j = blockIdx.x * kRouteThreads + tid; j < nlive; j += gridDim.x * kRouteThreads) {
                int lo = 0, hi = E - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (loff[mid] <= j)
                        lo = mid;
                    else
                        hi = mid - 1;
                }
                a.live_mtiles[j] = (poff[lo] >> 7) + (j - loff[lo]);
            }
        }
    }
    // padding rows of each expert's last tile: one warp per expert
    if (a.row_src) {
        for (int e = blockIdx.x * kRouteWarps + warp; e < E; e += gridDim.x * kRouteWarps)
            for (int r = poff[e] + cnt[e] + lane; r < poff[e + 1]; r += 32) {
                a.row_src[r] = -1;
                if (a.row_max) a.row_max[r] = a.row_max[a.rows_cap + r] = 0;
            }
    }

    // ---- phase 2: scatter this CTA's chunks
    int *wb = wbase + warp * E;
    int i_own = 0;
    for (int c = blockIdx.x; c < a.nchunks; c += gridDim.x, ++i_own) {
        const int wf0 = c * kRouteChunk + warp * kRouteSlice;
        int ids[kRouteIdsPerLane];
#pragma unroll
        for (int i = 0; i < kRouteIdsPerLane; ++i) {
            const int f = wf0 + 32 * i + lane;
            ids[i] = i_own == 0 ? ids_first[i] : f < a.R ? a.ids[f] : -1;  // valid here (checked above)
        }
        for (int e = lane; e < E; e += 32) wb[e] = 0;
        __syncwarp();
#pragma unroll
        for (int i = 0; i < kRouteIdsPerLane; ++i)
            if (ids[i] >= 0) atomicAdd(&wb[ids[i]], 1);
        __syncthreads();
        // each warp's first rank per expert: the chunk's rank plus the
        // earlier warps' counts
        for (int e = tid; e < E; e += kRouteThreads) {
            int run = cpre[i_own * E + e];
            for (int w = 0; w < kRouteWarps; ++w) {
                const int v = wbase[w * E + e];
                wbase[w * E + e] = run;
                run += v;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kRouteIdsPerLane; ++i) {
            const int f = wf0 + 32 * i + lane;
            const int e = ids[i];
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            const int pos = (e >= 0) ? wb[e] + rank : 0;
            __syncwarp();
            if (e >= 0 && rank == 0) wb[e] += __popc(peers);
            __syncwarp();
            if (e >= 0) {
                const int compact = off[e] + pos;
                const int padded = poff[e] + pos;
                a.row_of[f] = a.padded ? padded : compact;
                if (a.perm) a.perm[compact] = f;
                if (a.row_src) a.row_src[padded] = f;
                if (a.row_max) a.row_max[padded] = a.row_max[a.rows_cap + padded] = 0;
            }
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteArgs a)
{
    pdl_trigger();  // the quantiser may be scheduled; it waits for this kernel to finish
    pdl_wait();     // the scale check (status, reset barrier counter)
    route_body(a);
}

// The scale check and a one-CTA routing in one launch: the routing reads the
// status the check has just written, after a block barrier.
__global__ void __launch_bounds__(kRouteThreads) validate_route_kernel(ValidateArgs v, RouteArgs a)
{
    pdl_trigger();
    pdl_wait();  // whatever ran before on the stream (a previous call may still read the header)
    validate_body(v);
    __syncthreads();
    route_body(a);
}

// The scale check and the routing of a small batch (at most kTinyRouteRows
// routed rows, rows padded to 128 per expert) in one CTA: up to four routed
// rows per thread (row f = tid + 256 i), each row's rank among equal experts
// from a warp match within its 32-row step and the per-step counts, the
// offsets from one block scan.  The same outputs as route_body.
constexpr int kTinyRouteRowsPerThread = 4;
constexpr int kTinyRouteRows = kRouteThreads * kTinyRouteRowsPerThread;
__global__ void __launch_bounds__(kRouteThreads) validate_route_tiny_kernel(ValidateArgs v, RouteArgs a)
{
    extern __shared__ int sh[];
    __shared__ int s_bad;
    __shared__ int s_wsum[2][kRouteWarps];
    if (!a.trigger_after_wait) pdl_trigger();
    pdl_wait();  // whatever ran before on the stream (a previous call may still read the header)
    if (a.trigger_after_wait) pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, E = a.E;
    const int nsteps = (a.R + 31) >> 5;  // 32-row steps; step s holds rows [32 s, 32 s + 32)
    int id[kTinyRouteRowsPerThread];
#pragma unroll
    for (int i = 0; i < kTinyRouteRowsPerThread; ++i) {
        const int f = tid + kRouteThreads * i;
        id[i] = f < a.R ? a.ids[f] : -1;  // in flight during the scale check
    }
    int *wcnt = sh;                // [nsteps][E]: a step's rows per expert, then its first rank
    int *off = wcnt + nsteps * E;  // [E + 1]: counts, then compact offsets
    int *poff = off + E + 1;       // [E + 1]: padded offsets
    for (int i = tid; i < nsteps * E; i += kRouteThreads) wcnt[i] = 0;
    if (tid == 0) s_bad = 0;
    if (validate_body(v) != 0) return;  // (its block barriers order the clearing above)
    bool ok[kTinyRouteRowsPerThread];
    int wrank[kTinyRouteRowsPerThread];
#pragma unroll
    for (int i = 0; i < kTinyRouteRowsPerThread; ++i) {
        const int f = tid + kRouteThreads * i, step = f >> 5;
        const bool live = f < a.R;
        ok[i] = live && id[i] >= 0 && id[i] < E;
        if (live && !ok[i]) s_bad = 1;
        // (a step without a valid row skips the match: it costs about 0.3 us
        // a step, and small batches fill one or two steps of 32)
        wrank[i] = 0;
        if (__any_sync(0xffffffffu, ok[i])) {
            const unsigned peers = __match_any_sync(0xffffffffu, ok[i] ? id[i] : -1 - lane);
            wrank[i] = __popc(peers & ((1u << lane) - 1u));
            if (ok[i] && wrank[i] == 0) wcnt[step * E + id[i]] = __popc(peers);
        }
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            atomicOr(&a.hdr->error_flags, kErrBadExpertId);
            a.hdr->status = 3;  // nothing after this writes
        }
        return;
    }
    for (int e = tid; e < E; e += kRouteThreads) {
        int run = 0;
        for (int st = 0; st < nsteps; ++st) {
            const int c = wcnt[st * E + e];
            wcnt[st * E + e] = run;
            run += c;
        }
        off[e] = run;
    }
    __syncthreads();
    // exclusive scans of the counts and of the counts padded to 128 rows;
    // thread t owns experts [per t, per t + per)
    constexpr int kMaxPer = 1024 / kRouteThreads;
    const int per = (E + kRouteThreads - 1) / kRouteThreads, e0 = tid * per;
    int cl[kMaxPer], so = 0, sp = 0;
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) {
        const int e = e0 + i;
        cl[i] = (i < per && e < E) ? off[e] : 0;
        so += cl[i];
        sp += (cl[i] + 127) & ~127;
    }
    int io = so, ip = sp;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int to = __shfl_up_sync(0xffffffffu, io, o), tp = __shfl_up_sync(0xffffffffu, ip, o);
        if (lane >= o) {
            io += to;
            ip += tp;
        }
    }
    if (lane == 31) {
        s_wsum[0][warp] = io;
        s_wsum[1][warp] = ip;
    }
    __syncthreads();
    int xo = io - so, xp = ip - sp;
    for (int w = 0; w < warp; ++w) {
        xo += s_wsum[0][w];
        xp += s_wsum[1][w];
    }
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) {
        const int e = e0 + i;
        if (i < per && e < E) {
            off[e] = xo;
            poff[e] = xp;
        }
        xo += cl[i];
        xp += (cl[i] + 127) & ~127;
    }
    if (tid == kRouteThreads - 1) {
        off[E] = xo;
        poff[E] = xp;
    }
    __syncthreads();
    const int npad = poff[E];
    for (int e = tid; e <= E; e += kRouteThreads) {
        if (e < E) a.counts[e] = off[e + 1] - off[e];
        a.offsets[e] = off[e];
        a.pad_off[e] = poff[e];
        if (a.offsets_out) a.offsets_out[e] = off[e];
        if (e < E && a.tile_expert)
            for (int t = poff[e] >> 7; t < poff[e + 1] >> 7; ++t) a.tile_expert[t] = e;
    }
    if (tid == 0) {
        a.hdr->num_mtiles = npad >> 7;
        a.hdr->num_live_mtiles = npad >> 7;
    }
    // every padded row: no source (and UE8M0 row maxima 0); the routed rows'
    // sources are written after the barrier
    const int4 none = make_int4(-1, -1, -1, -1), zero = make_int4(0, 0, 0, 0);
    for (int r4 = tid; r4 < (npad >> 2); r4 += kRouteThreads) {
        if (a.row_src) reinterpret_cast<int4 *>(a.row_src)[r4] = none;
        if (a.row_max) {
            reinterpret_cast<int4 *>(a.row_max)[r4] = zero;
            reinterpret_cast<int4 *>(a.row_max + a.rows_cap)[r4] = zero;
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTinyRouteRowsPerThread; ++i) {
        if (!ok[i]) continue;
        const int f = tid + kRouteThreads * i;
        const int pos = wcnt[(f >> 5) * E + id[i]] + wrank[i];
        const int compact = off[id[i]] + pos, padded = poff[id[i]] + pos;
        a.row_of[f] = a.padded ? padded : compact;
        if (a.perm) a.perm[compact] = f;
        if (a.row_src) a.row_src[padded] = f;
    }
}

// ------------------------------------------------------------------ quantiser
// [page, §NVFP4 runtime-order figure; MoE section: SFScale[expert_idx]]:
// one warp per (token, 1024-element chunk), each lane two consecutive
// 16-element blocks.  The blocks' BF16 values and amax are read once and
// quantised for each of the token's k experts with that expert's global
// scale, into the expert's permuted row: 16 bytes of codes and two scale
// bytes per lane and expert.  Lane j < k loads expert j's destination row and
// global scale once per item and turns the row into the row's part of both
// output offsets; the expert loop broadcasts the three values by shuffle and
// adds the lane's own part, so it holds no per-row address arithmetic.
// Offsets are 32-bit (codes in 16-byte units, scales in bytes); the host
// keeps every call within that range.

constexpr int kQuantThreads = 128;  // 5 CTAs (20 warps) per SM at <= 96 registers

// SWZ: scales in the swizzled tensor-core layout (else linear [rows, H/16]);
// SF: block scales E4M3 (0) or UE8M0 bytes (1).  With UE8M0 and a row_max
// array, each routed row's largest scale byte is also recorded there
// (atomicMax; the array is zero on entry): the GEMM carries the row's bytes
// relative to it (ue8m0_carried).
//
// SELF (QuantArgs::self_route): the row map from the ids in shared memory.
// Expert e's rows start at 128 x (busy experts below e), in flat order; an id
// outside [0, E) gets no row.  The call's inputs were complete before this
// kernel could start (the one-CTA routing kernel lets it start only after its
// own dependency wait).
template <bool SWZ, int SF, bool SELF = false>
__global__ void __launch_bounds__(kQuantThreads, 5) quant_experts_kernel(QuantArgs a, DivTable tab_in)
{
    __shared__ DivTable2 tab;
    pdl_trigger();
    load_div_table(&tab, tab_in);
    const int *srow = nullptr;
    if constexpr (SELF) {
        static_assert(kQuantThreads >= kEarlyRows, "one routed row per thread");
        __shared__ int s_ids[kEarlyRows], s_row[kEarlyRows];
        __shared__ unsigned s_bits[32];
        __shared__ int s_wbase[32];
        const int R = a.T * a.k, f = threadIdx.x;
        if (f < 32) s_bits[f] = 0u;
        const int id = f < R ? ld_cg(a.ids + f) : -1;
        const bool ok = f < R && id >= 0 && id < a.E;
        if (f < R) s_ids[f] = id;
        __syncthreads();
        if (ok) atomicOr(&s_bits[id >> 5], 1u << (id & 31));
        __syncthreads();
        if (f < 32) {
            const int c = __popc(s_bits[f]);
            int incl = c;
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (f >= o) incl += v;
            }
            s_wbase[f] = incl - c;
        }
        __syncthreads();
        if (f < R) {
            int row = -1;
            if (ok) {
                int pos = 0;  // this expert's rows before f
                for (int j = 0; j < R; ++j) pos += (j < f && s_ids[j] == id) ? 1 : 0;
                row = 128 * (s_wbase[id >> 5] + __popc(s_bits[id >> 5] & ((1u << (id & 31)) - 1u))) + pos;
            }
            s_row[f] = row;
        }
        __syncthreads();
        srow = s_row;
    } else {
        __syncthreads();
        pdl_wait();  // the routing kernel's row map and status
        if (a.hdr && a.hdr->status != 0) return;
    }
    const int lane = threadIdx.x & 31;
    const int k = a.k, H = a.H;
    // blockIdx.y takes a share of each token's k experts: small batches spread
    // the expert loop over more CTAs instead of running it in one
    const int kper = (k + (int)gridDim.y - 1) / (int)gridDim.y;
    const int j0 = (int)blockIdx.y * kper, j1 = min(k, j0 + kper);
    const int npair = H >> 5;              // block pairs (32 elements) per row
    const int nchunk = (npair + 31) >> 5;  // warp items per row
    uint4 *const q16 = reinterpret_cast<uint4 *>(a.q);
    // items (t, c) = warp index + n * (warps in the grid), walked without dividing per item
    const int wpb = blockDim.x >> 5;
    const int warps = gridDim.x * wpb;
    const int w0 = blockIdx.x * wpb + (threadIdx.x >> 5);
    const int dt = warps / nchunk, dc = warps - dt * nchunk;
    int t = w0 / nchunk, c = w0 - (w0 / nchunk) * nchunk;
    while (t < a.T) {
        const int pair = c * 32 + lane;
        uint32_t my_q = 0, my_s = 0;  // lane j < k: row parts of expert j's code and scale offsets
        uint32_t my_row = 0;
        float my_g = 1.0f;
        bool my_ok = true;  // SELF: the row has a valid id
        if (lane < k) {
            const int f = t * k + lane;
            int srow_f = 0;
            if constexpr (SELF) {
                srow_f = srow[f];
                my_ok = srow_f >= 0;
                srow_f = max(srow_f, 0);
            }
            const uint32_t row = SELF ? (uint32_t)srow_f : (uint32_t)__ldg(a.row_of + f);
            my_row = row;
            if constexpr (SELF)
                my_g = my_ok ? __frcp_rn(ld_cg(a.in_scale + ld_cg(a.ids + f))) : 1.0f;
            else
                my_g = __ldg(a.g + __ldg(a.ids + f));
            my_q = row * (uint32_t)npair;
            my_s = SWZ ? ((row >> 7) * (uint32_t)a.sf_kc * 512u + (row & 31u) * 16u + ((row >> 5) & 3u) * 4u)
                       : row * (uint32_t)(H >> 4);
        }
        const bool active = pair < npair;
        const int b = 2 * pair;  // even: both scale bytes share one aligned 16-bit word
        const uint32_t lane_s = SWZ ? (uint32_t)(b >> 2) * 512u + (uint32_t)(b & 3) : (uint32_t)b;
        uint32_t w[16];
        if (active) {
            const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (size_t)t * H + (size_t)pair * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 v = SELF ? ld_cg(src + i) : __ldg(src + i);
                w[4 * i] = v.x;
                w[4 * i + 1] = v.y;
                w[4 * i + 2] = v.z;
                w[4 * i + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = 0u;
        }
        f32x2 x0[8], x1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x0[i] = bf16x2_to_f32x2(w[i]);
            x1[i] = bf16x2_to_f32x2(w[8 + i]);
        }
        const float amax0 = amax16_bf16(w), amax1 = amax16_bf16(w + 8);
        // not unrolled: the compact loop runs faster than eight inlined copies
#pragma unroll 1
        for (int j = j0; j < j1; ++j) {
            const uint32_t qo = __shfl_sync(0xffffffffu, my_q, j) + (uint32_t)pair;
            const uint32_t so = __shfl_sync(0xffffffffu, my_s, j) + lane_s;
            const float g = __shfl_sync(0xffffffffu, my_g, j);
            const bool okj = SELF ? __shfl_sync(0xffffffffu, my_ok ? 1 : 0, j) != 0 : true;
            uint32_t s0 = 0, s1 = 0;
            if (active && okj) {
                const uint2 p0 = SF ? quant_block16_ue8m0(x0, amax0, g, s0) : quant_block16(x0, amax0, g, &tab, s0);
                const uint2 p1 = SF ? quant_block16_ue8m0(x1, amax1, g, s1) : quant_block16(x1, amax1, g, &tab, s1);
                q16[qo] = make_uint4(p0.x, p0.y, p1.x, p1.y);
                *reinterpret_cast<uint16_t *>(a.sf + so) = (uint16_t)(s0 | (s1 << 8));
            }
            if (SF && a.row_max) {
                const uint32_t m = __reduce_max_sync(0xffffffffu, max(s0, s1));
                const uint32_t row = __shfl_sync(0xffffffffu, my_row, j);
                if (lane == 0) atomicMax(a.row_max + row, (int)m);
            }
        }
        t += dt;
        c += dc;
        if (c >= nchunk) {
            c -= nchunk;
            ++t;
        }
    }
    // SELF: this grid completes only after the routing kernel, so that the
    // next kernel's dependency wait covers both
    if constexpr (SELF) pdl_wait();
}

// ------------------------------------------------------------------ UE8M0 weight rows
// One warp per weight row (an output column of the GEMM): the row's largest
// UE8M0 block-scale byte m, stored as the row's factor 2^(c - 117) with the
// shift c = max(m - 18, 0) (see ue8m0_carried).
__global__ void __launch_bounds__(256) sf_row_factor_kernel(const uint8_t *sf, long long rows, int nsf,
                                                            float *row_factor)
{
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const uint8_t *src = sf + r * nsf;
        uint32_t m = 0;
        for (int i = lane; i < nsf; i += 32) m = max(m, (uint32_t)src[i]);
        m = __reduce_max_sync(0xffffffffu, m);
        if (lane == 0) row_factor[r] = ue8m0_row_factor(ue8m0_row_shift(m));
    }
}

// ------------------------------------------------------------------ weight-scale layout
// [page, "Kernel Backend": packed weights and scales are converted to the
// layout the chosen kernel wants].  One thread per output word (one row's four
// scales of a 64-element chunk), in 128x4-scale tiles of 128 rows x 64 K.
__global__ void __launch_bounds__(256) prep_sf_kernel(PrepArgs a)
{
    const int NT = a.N / 128;
    const long long total = (long long)a.E * NT * a.kc * 128;
    const int nsf = a.K / 16;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int v = (int)(i & 127);
        long long rest = i >> 7;
        const int c = (int)(rest % a.kc);
        rest /= a.kc;
        const int nt = (int)(rest % NT);
        const int e = (int)(rest / NT);
        // 128-row block nt of the expert.  w13: block 2t holds the gate rows
        // and block 2t+1 the up rows of h columns [128 t, 128 t + 128); when
        // I is an odd multiple of 64 the last block holds the final 64 gate
        // rows then the final 64 up rows.  Blocks of one tile are interleaved
        // per 64-K step, so a stage's scales are one contiguous run.
        int row;
        size_t blk_off;  // byte offset of (block, step c) within the expert
        if (a.gate_up_I > 0) {
            const int full = a.gate_up_I / 128;
            const int t = nt >> 1;
            if (t < full) {
                const int up = nt & 1;
                row = (up ? a.gate_up_I : 0) + 128 * t + v;
                blk_off = ((size_t)2 * t * a.kc + 2 * c + up) * 512;
            } else {
                row = v < 64 ? 128 * t + v : a.gate_up_I + 128 * t + (v - 64);
                blk_off = ((size_t)2 * t * a.kc + c) * 512;
            }
        } else {
            row = nt * 128 + v;
            blk_off = ((size_t)nt * a.kc + c) * 512;
        }
        const uint8_t *src = a.sf + ((size_t)e * a.N + row) * nsf;
        // UE8M0: carried relative to the row's largest byte (its shift read
        // back from the row factor that sf_row_factor_kernel wrote)
        const uint32_t shift = a.ue8m0 ? ue8m0_shift_of_factor(a.row_factor[(size_t)e * a.N + row]) : 0u;
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = 4 * c + j;
            if (col < nsf) word |= (a.ue8m0 ? ue8m0_carried(src[col], shift) : (uint32_t)src[col]) << (8 * j);
        }
        uint8_t *dst = a.out + (size_t)e * NT * a.kc * 512 + blk_off + (size_t)(v & 31) * 16 + (v >> 5) * 4;
        *reinterpret_cast<uint32_t *>(dst) = word;
    }
}

// ------------------------------------------------------------------ bounded waits
// The waits of the tensor-core kernels, made to run out: thread 0 waits on an
// mbarrier that nothing arrives on and gives up after limit_ns; thread 32
// waits on the same barrier with a limit ten times longer and gives up when
// thread 0 raises the CTA's abort flag.  Both record what happened in the
// status block as the GEMM kernels do (status 5 and their error bits).
__global__ void wait_selftest_kernel(DevHeader *hdr, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    volatile int *abort_v = &abort_flag;
    if (threadIdx.x == 0) {
        if (!tc::mbar_wait(&bar, 0, nullptr, limit_ns)) {
            *abort_v = 1;
            atomicOr(&hdr->error_flags, kErrTimeoutMma);
            hdr->status = 5;
        }
    } else if (threadIdx.x == 32) {
        if (!tc::mbar_wait(&bar, 0, abort_v, 10 * limit_ns)) atomicOr(&hdr->error_flags, kErrTimeoutEpilogue);
    }
}

// ------------------------------------------------------------------ residual + RMSNorm
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t *x, const float *out, int H, float eps,
                                                       uint16_t *xn)
{
    const int t = blockIdx.x;
    const uint16_t *xr = x + (size_t)t * H;
    const float *orow = out + (size_t)t * H;
    float ss = 0.0f;
    for (int i = threadIdx.x; i < H; i += blockDim.x) {
        const float r = __uint_as_float((uint32_t)xr[i] << 16) + orow[i];
        ss = fmaf(r, r, ss);
    }
    __shared__ float red[8];
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / (float)H + eps);
    __syncthreads();  // every thread has read `red` before x_next may overwrite x
    for (int i = threadIdx.x; i < H; i += blockDim.x) {
        const float r = __uint_as_float((uint32_t)xr[i] << 16) + orow[i];
        const float y = r * inv;
        uint32_t u = __float_as_uint(y);
        u += 0x7FFFu + ((u >> 16) & 1u);  // nearest BF16, ties to even (finite inputs)
        xn[(size_t)t * H + i] = (uint16_t)(u >> 16);
    }
}

// ------------------------------------------------------------------ static weight quantiser
// [page, glossary "Static weight quantization"; §NVFP4 two-level scale:
// 2688 = 6 * 448].  Pass 1: amax per tensor (non-negative floats order like
// their bit patterns, so an unsigned atomicMax is exact).
__global__ void __launch_bounds__(256) weight_amax_kernel(const uint16_t *w, long long per, unsigned *amax_bits)
{
    const int c = blockIdx.y;
    const uint16_t *src = w + (size_t)c * per;
    float m = 0.0f;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < per;
         i += (long long)gridDim.x * blockDim.x)
        m = fmaxf(m, fabsf(__uint_as_float((uint32_t)src[i] << 16)));
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) atomicMax(&amax_bits[c], __float_as_uint(m));
}

// Pass 2: weight_scale_2 = fl(amax / 2688), g = fl(1 / weight_scale_2), then
// the same block quantisation as activations.  A tensor of zeros has no
// usable scale: it gets weight_scale_2 = 0 (rejected by validation) and zero
// codes and scales.
template <bool UE>
__global__ void __launch_bounds__(256) weight_quant_kernel(const uint16_t *w, int N, int K, uint8_t *q,
                                                           uint8_t *sf, float *scale2,
                                                           const unsigned *amax_bits, DivTable tab_in)
{
    __shared__ DivTable2 tab;
    load_div_table(&tab, tab_in);
    __syncthreads();
    const int c = blockIdx.y;
    const float amax_t = __uint_as_float(amax_bits[c]);
    const float s2 = __fdiv_rn(amax_t, 2688.0f);
    const float g = __frcp_rn(s2);
    if (blockIdx.x == 0 && threadIdx.x == 0) scale2[c] = s2;
    const int nb = K >> 4;
    const long long total = (long long)N * nb;
    const uint16_t *src = w + (size_t)c * N * K;
    uint8_t *qc = q + (size_t)c * N * (K >> 1);
    uint8_t *sfc = sf + (size_t)c * N * nb;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(i / nb), b = (int)(i - (long long)n * nb);
        f32x2 x[8];
        float amax = 0.0f;
        const uint32_t *p = reinterpret_cast<const uint32_t *>(src + (size_t)n * K + (size_t)b * 16);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t wv = p[j];
            x[j] = bf16x2_to_f32x2(wv);
            amax = fmaxf(amax, fmaxf(fabsf(lo_f32(x[j])), fabsf(hi_f32(x[j]))));
        }
        uint32_t sb = 0;
        uint2 pk = make_uint2(0u, 0u);
        if (amax_t > 0.0f) pk = UE ? quant_block16_ue8m0(x, amax, g, sb) : quant_block16(x, amax, g, &tab, sb);
        *reinterpret_cast<uint2 *>(qc + (size_t)n * (K >> 1) + (size_t)b * 8) = pk;
        sfc[(size_t)n * nb + b] = (uint8_t)sb;
    }
}

int grid_for(long long work, int per_block, int waves_cap)
{
    long long g = (work + per_block - 1) / per_block;
    const long long cap = (long long)sm_count() * waves_cap;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

}  // namespace

cudaError_t launch_validate(const ValidateArgs &a, cudaStream_t st)
{
    const cudaError_t err = launch_pdl(validate_kernel, dim3(1), dim3(256), 0, st, a);
    return err != cudaSuccess ? err : cudaGetLastError();
}

namespace {
// Routing launch shape: a cooperative grid of at most as many CTAs as can be
// resident at once, each taking every gridDim-th chunk.
// per-step counts for R routed rows, and the two offset arrays
size_t tiny_route_smem(int R, int E) { return sizeof(int) * ((size_t)((R + 31) / 32) * E + 2 * ((size_t)E + 1)); }
constexpr size_t kTinyRouteSmemMax = 96 * 1024;

size_t route_smem(int E)
{
    // cnt, off, poff, per-warp bases, per-chunk prefixes, per-run sums, live-tile offsets
    return sizeof(int) *
           ((4 + kRouteWarps + kRouteMaxOwn) * (size_t)E + 3 + (E > kRouteThreads ? E : kRouteThreads));
}

cudaError_t route_plan(const RouteArgs &a, int *grid_out)
{
    static int resident[64] = {0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!resident[dev]) {
        // sized once for the largest expert count, so any call fits
        const size_t smem_max = route_smem(1024);
        err = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(validate_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
        if (err != cudaSuccess) return err;
        int per_sm = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_kernel, kRouteThreads, smem_max);
        if (err != cudaSuccess) return err;
        resident[dev] = (per_sm < 1 ? 1 : per_sm) * sm_count();
    }
    int grid = a.nchunks < resident[dev] ? a.nchunks : resident[dev];
    if (grid < 1) grid = 1;
    if ((a.nchunks + grid - 1) / grid > kRouteMaxOwn) return cudaErrorInvalidConfiguration;
    *grid_out = grid;
    return cudaSuccess;
}
}  // namespace

cudaError_t launch_route(const RouteArgs &a, cudaStream_t st)
{
    int grid = 0;
    const cudaError_t err = route_plan(a, &grid);
    if (err != cudaSuccess) return err;
    const size_t smem = route_smem(a.E);
    RouteArgs args = a;
    if (grid == 1) {
        // one CTA: no grid barrier, so a plain launch (which may overlap the
        // scale check's tail) does
        const cudaError_t e = launch_pdl(route_kernel, dim3(1), dim3(kRouteThreads), smem, st, args);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    void *params[] = {&args};
    return cudaLaunchCooperativeKernel((const void *)route_kernel, dim3(grid), dim3(kRouteThreads), params, smem, st);
}

cudaError_t launch_validate_route(const ValidateArgs &v, const RouteArgs &a, cudaStream_t st)
{
    if (a.R <= kTinyRouteRows && a.pad_rows != 256 && !a.live_mtiles && tiny_route_smem(a.R, a.E) <= kTinyRouteSmemMax) {
        static bool attr_set[64] = {false};
        int dev = 0;
        cudaError_t err = cudaGetDevice(&dev);
        if (err != cudaSuccess) return err;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!attr_set[dev]) {
            err = cudaFuncSetAttribute(validate_route_tiny_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kTinyRouteSmemMax);
            if (err != cudaSuccess) return err;
            attr_set[dev] = true;
        }
        err = launch_pdl(validate_route_tiny_kernel, dim3(1), dim3(kRouteThreads), tiny_route_smem(a.R, a.E), st, v,
                         a);
        return err != cudaSuccess ? err : cudaGetLastError();
    }
    if (a.trigger_after_wait) return cudaErrorInvalidValue;  // the one-CTA form only
    int grid = 0;
    cudaError_t err = route_plan(a, &grid);
    if (err != cudaSuccess) return err;
    if (grid > 1) {
        err = launch_validate(v, st);
        return err != cudaSuccess ? err : launch_route(a, st);
    }
    err = launch_pdl(validate_route_kernel, dim3(1), dim3(kRouteThreads), route_smem(a.E), st, v, a);
    return err != cudaSuccess ? err : cudaGetLastError();
}

cudaError_t launch_quant_experts(const QuantArgs &a, cudaStream_t st)
{
    const long long work = (long long)a.T * ((a.H / 32 + 31) / 32) * 32;  // one lane per block pair
    // One full wave of resident CTAs, grid-striding over the work.
    auto launch = [&](auto kernel) {
        int per_sm = 1;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kQuantThreads, 0) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        const long long wave = (long long)sm_count() * per_sm;
        long long grid = wave;
        const long long need = (work + kQuantThreads - 1) / kQuantThreads;
        if (grid > need) grid = need;
        if (grid < 1) grid = 1;
        // a batch that fills less than a wave splits each token's experts
        // over gridDim.y, up to one expert per CTA
        long long ysplit = wave / grid;
        if (ysplit > a.k) ysplit = a.k;
        if (ysplit < 1) ysplit = 1;
        return launch_pdl(kernel, dim3((int)grid, (int)ysplit), dim3(kQuantThreads), 0, st, a, div_table());
    };
    cudaError_t err;
    if (a.self_route) {
        // E4M3, swizzled, a padded row map of at most kEarlyRows routed rows
        if (a.sf_ue8m0 || !a.sf_swizzled || (long long)a.T * a.k > kEarlyRows || !a.in_scale)
            return cudaErrorInvalidValue;
        err = launch(quant_experts_kernel<true, 0, true>);
    } else if (a.sf_ue8m0)
        err = a.sf_swizzled ? launch(quant_experts_kernel<true, 1>) : launch(quant_experts_kernel<false, 1>);
    else
        err = a.sf_swizzled ? launch(quant_experts_kernel<true, 0>) : launch(quant_experts_kernel<false, 0>);
    return err != cudaSuccess ? err : cudaGetLastError();
}

cudaError_t launch_prep_sf(const PrepArgs &a, cudaStream_t st)
{
    if (a.ue8m0) {
        const long long rows = (long long)a.E * a.N;
        sf_row_factor_kernel<<<grid_for(rows * 32, 256, 16), 256, 0, st>>>(a.sf, rows, a.K / 16, a.row_factor);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const long long work = (long long)a.E * (a.N / 128) * a.kc * 128;
    prep_sf_kernel<<<grid_for(work, 256, 16), 256, 0, st>>>(a);
    return cudaGetLastError();
}

// Every (byte b, row shift c) pair through both carry routines: out[c][b] by
// ue8m0_carried, out[256 + c][b] by ue8m0_carried4 (four bytes a word).
__global__ void ue8m0_carry_selftest_kernel(uint8_t *out)
{
    const uint32_t c = blockIdx.x, b = threadIdx.x;
    out[c * 256 + b] = (uint8_t)ue8m0_carried(b, c);
    if ((b & 3) == 0) {
        const uint32_t w = b | (b + 1) << 8 | (b + 2) << 16 | (b + 3) << 24;
        *reinterpret_cast<uint32_t *>(out + (256 + c) * 256 + b) = ue8m0_carried4(w, c * 0x01010101u);
    }
}
cudaError_t launch_ue8m0_carry_selftest(uint8_t *out, cudaStream_t st)
{
    ue8m0_carry_selftest_kernel<<<256, 256, 0, st>>>(out);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(DevHeader *hdr, uint64_t limit_ns, cudaStream_t st)
{
    wait_selftest_kernel<<<1, 64, 0, st>>>(hdr, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const uint16_t *x, const float *out, int T, int H, float eps, uint16_t *xn,
                           cudaStream_t st)
{
    rmsnorm_kernel<<<T, 256, 0, st>>>(x, out, H, eps, xn);
    return cudaGetLastError();
}

cudaError_t launch_quantize_weights(const uint16_t *w, int count, int N, int K, uint8_t *q, uint8_t *sf,
                                    float *scale2, unsigned *amax_bits, int ue8m0, cudaStream_t st)
{
    cudaError_t err = cudaMemsetAsync(amax_bits, 0, sizeof(unsigned) * (size_t)count, st);
    if (err != cudaSuccess) return err;
    const long long per = (long long)N * K;
    dim3 g1(grid_for(per, 256 * 8, 4), count);
    weight_amax_kernel<<<g1, 256, 0, st>>>(w, per, amax_bits);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    dim3 g2(grid_for((long long)N * (K / 16), 256, 4), count);
    if (ue8m0)
        weight_quant_kernel<true><<<g2, 256, 0, st>>>(w, N, K, q, sf, scale2, amax_bits, div_table());
    else
        weight_quant_kernel<false><<<g2, 256, 0, st>>>(w, N, K, q, sf, scale2, amax_bits, div_table());
    return cudaGetLastError();
}

}  // namespace nvfp4
