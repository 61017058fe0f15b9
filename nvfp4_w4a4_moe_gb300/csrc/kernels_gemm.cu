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
// Kernel shape (one persistent CTA per SM):
//   warp 0     TMA producer: per 256-K stage the A tile (128 rows, 128-byte
//              swizzle), the B tile, and the 128x4-scale tiles of both (plain
//              bulk copies) into a 4-stage ring; for w2 the A tile goes to a
//              ring of five slots of its own, once per pair of tiles.
//   warp 1     TMEM owner (512 columns) and MMA issuer: per stage, 4 x
//              tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (K64):
//              M128 N256 into one accumulator (w13), M128 N128 into one of two
//              (w2).
//   epilogue   8 (w13) or 16 (w2) warps, two or four per TMEM lane quarter:
//              tcgen05.ld of the accumulator, released before the heavy work,
//              then either SiLU(gate)*up + NVFP4 requantisation (w13) or the
//              weighted scatter-add into the token-order output (w2),
//              transposed through shared memory so the FP32 reductions are
//              coalesced.
//   last 4     scale writers, one per TMEM lane quarter: per stage they move
//              both operands' scale tiles smem -> registers -> TMEM
//              (tcgen05.st).
// Every wait is bounded (%globaltimer); on expiry the kernel records the
// error in the workspace header, drains what it has in flight and exits.
#include <climits>

#include "internal.h"
#include "tc_common.cuh"

namespace nvfp4 {
namespace {

using namespace tc;

constexpr int BM = 128, BK = 256;  // BK in FP4 elements (128 bytes per row)
constexpr int A_BYTES = BM * BK / 2;
constexpr int SF_TILE = 512;                 // one 128x4-scale tile: 128 rows x 64 K
constexpr int SFA_BYTES = 4 * SF_TILE;       // 256 K per stage
constexpr int TMEM_COLS = 512;
constexpr int NUM_SCALE_WARPS = 4;  // one per TMEM lane quarter
// Row of the per-warp 32 x 32 transpose buffer: 32 floats in eight 16-byte
// chunks, logical chunk j of row r stored at chunk j ^ (r & 7).  A row written
// by one lane and four rows read by 8 lanes each are then 128-bit accesses
// that take the minimum four wavefronts.
constexpr int XPOSE_LD = 32;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;

// Per-kernel plan.
//  w13: tiles of 128 rows x (128 gate + 128 up) columns, one M128 N256 MMA per
//       64-K step (the last tile of an I that is an odd multiple of 64 is
//       64 gate + 64 up wide, N128).  The 256-column FP32 accumulator leaves no
//       TMEM for a second one, so the epilogue copies it to registers and
//       releases it before computing; a 4-stage ring of 54 KB stages.
//       Eight epilogue warps, two per TMEM lane quarter.
//  w2:  tiles of 128 x 128, M128 N128 MMAs into two alternating accumulators,
//       a 4-stage ring of B and scales, A in three slots of its own (one per
//       256-K stage) filled once per pair of tiles that share the m-tile (two
//       adjacent output column blocks, run back to back), and sixteen
//       epilogue warps in two groups of eight that
//       take alternate tiles (one accumulator each), so one group is issuing
//       the combine's reductions while the other waits on TMEM and fetches
//       its rows' tokens and weights; each warp has a transpose buffer.
//  w13, CTA2: the same tiles computed by a pair of CTAs (a cluster of two) on
//       two m-tiles of one expert: one M256 N256 MMA per 64-K step
//       (tcgen05 .cta_group::2, issued by rank 0).  Each CTA loads its own
//       m-tile's A and scales, half of B (rank 0 the gate rows, rank 1 the up
//       rows) and all of B's scales (the pair MMA reads the B scales of all N
//       from each CTA's tensor memory); its accumulator holds its 128 rows.
//       38 KB per stage per CTA instead of 54, a 5-stage ring, and sixteen
//       epilogue warps.
//  w13, small batches (at most kSmallPlanRows routed rows, so that no
//       m-tile holds more): tiles of 64 h columns (64 gate + 64 up weight
//       rows, N128; the B scales cut from the block's two 128-row scale
//       tiles), the A stage only the m-tile's first kSmallPlanRows rows, and a
//       7-stage ring.  At these sizes a tile's K loop is paced by the ring's
//       round trip, not by its bytes: more stages in flight, on twice the
//       tiles.
//  w2, small batches (at most kSmallPlanRowsW2 routed rows): A in the ring
//       (an m-tile's first kSmallPlanRowsW2 rows, no tile pairs), a 7-stage
//       ring, and the combine added from registers (a tile holds one or two
//       live rows; no transpose buffer).
//  w13, small batches where every CTA holds one tile (QA): the small-batch
//       plan with A quantised in the kernel.  The epilogue warps, idle until
//       the first accumulator, quantise the m-tile's rows (the quantiser's
//       block routine) into a persistent buffer of all its K slices, in the
//       layout a TMA 128-byte-swizzled load leaves, and their scales into
//       persistent scale tiles; the producer streams only the weights, and
//       the a1 quantiser launch goes.  A 6-stage ring.  The CTA also routes
//       its own tile from the call's ids (at most 32 routed rows: one m-tile
//       per busy expert, in expert order, rows in flat order, as the routing
//       kernel lays them out) and forms its expert's scales from the input and
//       weight scales as the scale check does, so that the loads, the A
//       quantisation and the MMAs need nothing the routing kernel writes and
//       run before the dependency wait; the epilogue's writes come after it,
//       and only when the scale check and routing passed.
constexpr int kDecRows = (int)kSmallPlanRows, kDecRowsW2 = (int)kSmallPlanRowsW2;
static_assert(kDecRows % 16 == 0 && kDecRowsW2 % 16 == 0, "A is loaded in 16-row boxes");
constexpr int kQaSlices = (int)kInlineQuantMaxK / BK;  // K slices of the persistent A buffer
template <int EPI, bool CTA2 = false, bool DEC = false, bool QA = false, bool EARLY = false>
struct Plan {
    static constexpr int DEC_ROWS = EPI == 0 ? kDecRows : kDecRowsW2;  // small-batch plan: A rows per stage
    static constexpr int BN = DEC ? 128 : EPI == 0 ? 256 : 128;  // widest tile (MMA N)
    static constexpr int STAGES = QA ? 6 : DEC ? 7 : CTA2 ? 5 : 4;
    // w13 pairs: 16 epilogue warps of 32 columns each, so every warp releases
    // the accumulator after a single TMEM load (the pair form's stages are
    // shorter, and the release gates the next tile's MMAs); 8 for w13 on
    // single CTAs, where 16 measured no faster
    static constexpr int NUM_EPI_WARPS = EPI == 0 ? (CTA2 ? 16 : 8) : 16;
    static constexpr int EPI_THREADS = 32 * NUM_EPI_WARPS;
    static constexpr int EPI_GROUPS = EPI == 0 ? 1 : 2;  // w2: one group of eight warps per accumulator
    static constexpr int SCALE_WARP0 = 2 + NUM_EPI_WARPS;  // then the four scale writers
    static constexpr int NUM_THREADS = 64 + EPI_THREADS + 32 * NUM_SCALE_WARPS;
    static constexpr int ACC_BUFS = EPI == 0 ? 1 : 2;
    static constexpr int B_BYTES = (CTA2 ? BN / 2 : BN) * BK / 2;  // B rows this CTA loads per stage
    // w2: A lives in a ring of slots of its own, outside the B ring, so that a
    // tile pair (two column blocks of one m-tile) loads it once.  Fill f (one
    // 256-K stage of one m-tile) takes slot f % A_SLOTS and completes on the
    // B ring stage it is issued with.  No barrier of its own is needed: before
    // fill f + A_SLOTS is issued the producer has waited for the MMAs of a ring
    // stage at or after the last one reading fill f (checked for every K depth
    // a pair can have, 1 .. A_SLOTS stages, and for unpaired tiles).
    static constexpr int A_SLOTS = EPI == 1 && !DEC ? 5 : 0;
    // A ring stages sit A_STRIDE apart; the MMA reads 128 rows from each
    // stage's start, so in the small-batch plan the rows past the loaded ones
    // read the following stages (their outputs are never stored), and the
    // region ends a full A tile after the last stage's start
    static constexpr int A_STRIDE = DEC ? DEC_ROWS * BK / 2 : A_BYTES;
    static constexpr int RING_A_REGION =
        A_SLOTS > 0 ? 0 : ((QA ? kQaSlices : STAGES) - 1) * A_STRIDE + A_BYTES;  // QA: the persistent A slices
    static constexpr int SFA_REGION = (QA ? kQaSlices : STAGES) * SFA_BYTES;      // QA: persistent A scale tiles
    static constexpr int SFB_BYTES = DEC && EPI == 0 ? 2 * 4 * SF_TILE : (BN / 128) * 4 * SF_TILE;
    static constexpr int SFB_STEP = BN / 32;               // TMEM columns per 64-K step of B scales
    static constexpr int SF_COLS = 16 + 4 * SFB_STEP;      // TMEM scale columns per stage
    static constexpr int SF_TMEM_COL = ACC_BUFS * BN;      // scale slots after the accumulator(s)
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + RING_A_REGION;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SFB = OFF_SFA + SFA_REGION;
    static constexpr int OFF_AS = OFF_SFB + STAGES * SFB_BYTES;  // the A slots (w2)
    static constexpr int OFF_BAR = OFF_AS + A_SLOTS * A_BYTES;
    static constexpr int NUM_BARS = 3 * STAGES + 2 * ACC_BUFS + 2;  // + drain, QA's A-ready
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    // the CTA's own routing: QaRoute (QA) or EarlyRoute (w13 on single CTAs)
    static constexpr int OFF_QAR = (OFF_MISC + 16 + 15) & ~15;
    static constexpr int QAR_BYTES = QA ? 256 : (EARLY || (EPI == 1 && DEC)) ? 1024 : 0;  // (w2 small: the tile map)
    static constexpr int OFF_XPOSE = (OFF_QAR + QAR_BYTES + 15) & ~15;
    static constexpr int XPOSE_BYTES = EPI == 1 && !DEC ? NUM_EPI_WARPS * 32 * XPOSE_LD * 4 : 0;
    static constexpr int SMEM_BYTES = OFF_XPOSE + XPOSE_BYTES + 1024;  // + alignment slack
    static_assert(SF_TMEM_COL + STAGES * SF_COLS <= TMEM_COLS, "scale slots exceed TMEM");
    static_assert(EPI_GROUPS == ACC_BUFS, "each epilogue group owns one accumulator");
    static_assert(OFF_B % 1024 == 0 && OFF_AS % 1024 == 0, "128-byte-swizzled operands start on 1024 bytes");
    static_assert(EPI == 0 || DEC || (A_SLOTS == 5 && STAGES == 4), "the A-slot reuse argument is for 5 slots, 4 stages");
    static_assert(!CTA2 || EPI == 0, "CTA pairs: w13 only");
    static_assert(!DEC || !CTA2, "the small-batch plans: single CTAs");
    static_assert(!QA || (DEC && EPI == 0 && DEC_ROWS == 32), "A quantised in the kernel: w13's small-batch plan");
    static_assert(!EARLY || (!CTA2 && !QA && (EPI == 0 ? !DEC : DEC)),
                  "early weights: w13's wide tiles, w2's small-batch plan, single CTAs");
    static_assert(SMEM_BYTES + (EPI == 0 ? (int)sizeof(DivTable2) : 0) <= 232448,
                  "shared memory plan exceeds the opt-in limit");
};

// Instruction descriptor, block-scaled kinds: E2M1 A and B (code 1 at bits
// 7-9 and 10-12), K-major both, N>>3 at 17-22, scale type UE4M3 (bit 23 = 0),
// M>>4 at 24-28, scale-factor ids 0.
__host__ __device__ constexpr uint32_t idesc_for(int n, int m = BM)
{
    return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
}
// The pair's form (.cta_group::2, M256): A from both CTAs' shared memory at
// the same offsets (128 rows each), B half from each, D and the scale
// factors in each CTA's tensor memory at the same addresses.
__device__ __forceinline__ void tc_mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
}

// ---------------------------------------------------------------- tiles
// Tile geometry shared by every role.  w13: tile t covers h columns
// [128 t, 128 t + hc) with hc = min(128, I - 128 t); its B rows are hc gate
// rows then hc up rows, and its weight scales are hc*2/128 tiles per 64-K
// step.  w2: tile t covers output columns [128 t, 128 t + 128).
template <int EPI>
struct TileInfo {
    int mt, nt, e;
    int hc;       // w13: h columns of the tile (128 or 64)
    int hc0;      // w13: its first h column
    int nblk;     // 128-row scale tiles per 64-K step of the tile's scale block (w13 full block: 2, else 1)
    int compose;  // w13 64-column tile cut from a full block: 1 + which half of its two tiles; else 0
};
// QA: the CTA's own tile, routed from the call's ids in the prologue (one
// warp), and its expert's scales.
struct QaRoute {
    int f[32];           // the m-tile's live rows: their flat indices t * k + j, in order
    int e;               // the tile's expert; -1: no tile for this CTA
    int mt, nt;          // m-tile (the expert's rank among the busy experts) and 64-column tile
    int nlive;           // live rows of the m-tile
    int mtiles;          // busy experts: one m-tile each
    int bad;             // an id outside [0, E) (the routing kernel refuses the call)
};
static_assert(sizeof(QaRoute) <= 256, "QA routing block");

// Up to 32 routed rows (one per lane): each busy expert holds one m-tile (at
// most 32 rows of 128), m-tiles in ascending expert order, an expert's rows in
// ascending flat index: the layout the routing kernel writes.
__device__ __forceinline__ void qa_route(const GemmArgs &p, QaRoute *q, int lane)
{
    const unsigned full = 0xffffffffu;
    int id = lane < p.R ? ld_cg(p.ids + lane) : -1;
    const bool live = lane < p.R && id >= 0 && id < p.E;
    const bool anybad = __ballot_sync(full, lane < p.R && !live) != 0u;
    if (!live) id = -1;
    const unsigned peers = __match_any_sync(full, live ? id : -1 - lane);
    const bool first = live && __ffs(peers) - 1 == lane;  // the expert's first row
    int rank = 0;  // busy experts below this row's
    for (int j = 0; j < 32; ++j) {
        const int idj = __shfl_sync(full, id, j);
        const int fj = __shfl_sync(full, first ? 1 : 0, j);
        rank += (fj != 0 && idj < id) ? 1 : 0;
    }
    const unsigned firsts = __ballot_sync(full, first);
    const int NTq = (p.gate_up_I + 63) / 64;
    const int mt = (int)blockIdx.x / NTq, nt = (int)blockIdx.x - mt * NTq;
    const unsigned hit = __ballot_sync(full, first && rank == mt);
    const int eid = __shfl_sync(full, id, hit ? __ffs(hit) - 1 : 0);
    const int e = (hit != 0u && !anybad) ? eid : -1;
    const unsigned rows = __ballot_sync(full, live && id == e);
    if ((rows >> lane) & 1u) q->f[__popc(rows & ((1u << lane) - 1u))] = lane;
    if (lane == 0) {
        q->e = e;
        q->mt = mt;
        q->nt = nt;
        q->nlive = __popc(rows);
        q->mtiles = __popc(firsts);
        q->bad = anybad ? 1 : 0;
    }
}

// w2 walks the m-tiles that hold rows (live_mtiles, when the rows are padded
// to 256 for the paired w13) in order.
__device__ __forceinline__ int mtile_of(const GemmArgs &p, int mi) { return p.live_mtiles ? p.live_mtiles[mi] : mi; }

// W: w13 tile width in h columns (128, or 64 in the small-batch plan).  The
// tile's scales are those of the 128-column block holding it: per 64-K step
// a gate and an up 128-row tile (a full block), or one tile of 64 gate + 64
// up rows (the last block when I is an odd multiple of 64).
// STE: the tile map is read from a shared-memory copy `ste` instead of memory.
template <int EPI, bool STE = false>
__device__ __forceinline__ TileInfo<EPI> tile_info(const GemmArgs &p, int tile, int NT, int MT, int W = 128,
                                                   const int *ste = nullptr)
{
    TileInfo<EPI> ti;
    if (EPI == 0) {
        // m-tile major: the CTAs working at one time share a few A tiles
        ti.mt = tile / NT;
        ti.nt = tile - ti.mt * NT;
    } else {
        // column-block major: at any time the combine's reductions touch one or
        // two 128-column blocks of `out` (4 MB at 8192 tokens), which stay in
        // L2 instead of being evicted and re-read from HBM between the k
        // contributions to each row; an expert's m-tiles stay adjacent, so its
        // B tile is reused from L2
        ti.nt = tile / MT;
        ti.mt = mtile_of(p, tile - ti.nt * MT);
    }
    ti.e = STE ? ste[ti.mt] : p.tile_expert[ti.mt];
    if (EPI == 0) {
        ti.hc0 = W * ti.nt;
        ti.hc = min(W, p.gate_up_I - ti.hc0);
        const bool full_block = (ti.hc0 & ~127) + 128 <= p.gate_up_I;
        ti.nblk = full_block ? 2 : 1;
        ti.compose = W == 64 && full_block ? 1 + (ti.nt & 1) : 0;
    } else {
        ti.hc = ti.hc0 = ti.compose = 0;
        ti.nblk = 1;
    }
    return ti;
}

// The CTA's i-th tile.  w13, and w2 when a tile pair does not fit the A
// slots: tile blockIdx + i * gridDim of tile_info's order.  w2 paired: units
// (m-tile, pair of adjacent output column blocks) in column-pair-major order,
// unit (i/2) * gridDim + blockIdx, column block 2 * pair + (i & 1); the two
// tiles of a unit run back to back and share the A operand.
template <int EPI, bool CTA2 = false, bool STE = false>
__device__ __forceinline__ TileInfo<EPI> seq_tile(const GemmArgs &p, int i, int NT, int MT, bool paired, int W,
                                                  const int *ste = nullptr)
{
    if (CTA2) {
        // unit (m-tile pair, column tile), pair-major; this CTA's m-tile of the pair
        const int G = (int)gridDim.x >> 1, b = (int)blockIdx.x >> 1;
        TileInfo<EPI> ti = tile_info<EPI>(p, b + i * G, NT, MT);
        ti.mt = 2 * ti.mt + (int)(blockIdx.x & 1);
        ti.e = p.tile_expert[ti.mt];
        return ti;
    }
    if (EPI == 1 && paired) {
        const int u = (i >> 1) * (int)gridDim.x + (int)blockIdx.x;
        const int g = u / MT;
        TileInfo<EPI> ti;
        ti.mt = mtile_of(p, u - g * MT);
        ti.nt = 2 * g + (i & 1);
        ti.e = p.tile_expert[ti.mt];
        ti.hc = ti.hc0 = ti.compose = 0;
        ti.nblk = 1;
        return ti;
    }
    return tile_info<EPI, STE>(p, (int)blockIdx.x + i * (int)gridDim.x, NT, MT, W, ste);
}

// Early weights (w13, at most kEarlyRows routed rows): the busy experts of
// the call's ids, in ascending order.  Each holds one m-tile (at most 128
// rows), in that order: the routing kernel's tile map.
struct EarlyRoute {
    unsigned bits[32];  // busy-expert bitmap (E <= 1024)
    int busy[kEarlyRows];
    int mtiles;
    int bad;            // an id outside [0, E) (the routing kernel refuses the call)
};
static_assert(sizeof(EarlyRoute) <= 1024, "early routing block");

__device__ __forceinline__ void early_route(const GemmArgs &p, EarlyRoute *q, int lane)
{
    const unsigned full = 0xffffffffu;
    q->bits[lane] = 0u;
    __syncwarp();
    bool bad = false;
    for (int f = lane; f < p.R; f += 32) {
        const int id = ld_cg(p.ids + f);
        if (id >= 0 && id < p.E)
            atomicOr(&q->bits[id >> 5], 1u << (id & 31));
        else
            bad = true;
    }
    __syncwarp();
    const unsigned w = q->bits[lane];
    const int c = __popc(w);
    int incl = c;
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(full, incl, o);
        if (lane >= o) incl += v;
    }
    int pos = incl - c;
    for (unsigned m = w; m != 0u && pos < kEarlyRows; m &= m - 1u) q->busy[pos++] = 32 * lane + __ffs(m) - 1;
    const bool anybad = __any_sync(full, bad || p.R > kEarlyRows);  // (the host keeps R within kEarlyRows)
    if (lane == 31) q->mtiles = incl;
    if (lane == 0) q->bad = anybad ? 1 : 0;
}

// QA: the tile qa_route chose (w13, 64-column tiles)
template <int EPI>
__device__ __forceinline__ TileInfo<EPI> qa_tile(const GemmArgs &p, const QaRoute *q)
{
    TileInfo<EPI> ti;
    ti.mt = q->mt;
    ti.nt = q->nt;
    ti.e = q->e;
    ti.hc0 = 64 * ti.nt;
    ti.hc = min(64, p.gate_up_I - ti.hc0);
    const bool full_block = (ti.hc0 & ~127) + 128 <= p.gate_up_I;
    ti.nblk = full_block ? 2 : 1;
    ti.compose = full_block ? 1 + (ti.nt & 1) : 0;
    return ti;
}

// Early weights: tile t of tile_info's order (w13 m-tile major, w2 column
// block major), its expert from the early route instead of the routing
// kernel's tile map.
template <int EPI>
__device__ __forceinline__ TileInfo<EPI> early_tile(const GemmArgs &p, const EarlyRoute *q, int t, int NT, int MT,
                                                    int W)
{
    TileInfo<EPI> ti;
    if (EPI == 0) {
        ti.mt = t / NT;
        ti.nt = t - ti.mt * NT;
    } else {
        ti.nt = t / MT;
        ti.mt = t - ti.nt * MT;
    }
    ti.e = q->busy[ti.mt];
    if (EPI == 0) {
        ti.hc0 = W * ti.nt;
        ti.hc = min(W, p.gate_up_I - ti.hc0);
        const bool full_block = (ti.hc0 & ~127) + 128 <= p.gate_up_I;
        ti.nblk = full_block ? 2 : 1;
        ti.compose = W == 64 && full_block ? 1 + (ti.nt & 1) : 0;
    } else {
        ti.hc = ti.hc0 = ti.compose = 0;
        ti.nblk = 1;
    }
    return ti;
}

// Early weights: the A loads of the first n ring stages (stage s holds load
// s of the CTA's sequence: tile b + (s / KT) * G, K step s % KT), issued once
// the dependency wait has returned.
template <int EPI, class P, bool DEC>
__device__ __forceinline__ void early_a_loads(const GemmArgs &p, uint8_t *smem, uint64_t *full, const CUtensorMap *ta,
                                              const CUtensorMap *ta16, int n, int b, int G, int NT, int MT, int KT)
{
    for (int s = 0; s < n; ++s) {
        const int t = b + (s / KT) * G, kt = s % KT;
        const int mt = EPI == 0 ? t / NT : t % MT;
        const int kx = kt * (BK / 2);
        if constexpr (DEC) {
            for (int r = 0; r < P::DEC_ROWS; r += 16)
                tma_2d(smem + P::OFF_A + s * P::A_STRIDE + r * (BK / 2), ta16, kx, mt * BM + r, &full[s]);
        } else {
            tma_2d(smem + P::OFF_A + s * A_BYTES, ta, kx, mt * BM, &full[s]);
        }
        bulk_g2s(smem + P::OFF_SFA + s * SFA_BYTES, p.a_sf + ((size_t)mt * p.a_kc + 4 * kt) * SF_TILE, SFA_BYTES,
                 &full[s]);
    }
}

// ---------------------------------------------------------------- kernel
// EPI 0: w13 (SiLU*up + requantise), 1: w2 (weighted combine).  UE: UE8M0
// block scales throughout.  The A scales arrive as UE8M0 bytes and are
// carried to the tensor cores per row (ue8m0_carried, with the row's largest
// byte from a_row_max); the weight scales were carried per weight row when
// prepared.  The epilogue multiplies both rows' factors back: the A row's
// into the row scale, the weight row's per output column.  w13 then writes
// a2 as UE8M0 bytes with each row's largest byte (out_row_max).
template <int EPI, bool UE, bool CTA2, bool DEC, bool QA, bool EARLY>
__global__ void __launch_bounds__(Plan<EPI, CTA2, DEC, QA, EARLY>::NUM_THREADS, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_a16, const GemmArgs p, const DivTable tab_in)
{
    using P = Plan<EPI, CTA2, DEC, QA, EARLY>;
    constexpr int STAGES = P::STAGES, ACC_BUFS = P::ACC_BUFS, OFF_A = P::OFF_A, OFF_B = P::OFF_B,
                  OFF_SFA = P::OFF_SFA, OFF_SFB = P::OFF_SFB, OFF_BAR = P::OFF_BAR, OFF_MISC = P::OFF_MISC,
                  OFF_XPOSE = P::OFF_XPOSE, B_BYTES = P::B_BYTES, SFB_BYTES = P::SFB_BYTES,
                  SFB_STEP = P::SFB_STEP, SF_COLS = P::SF_COLS, SF_TMEM_COL = P::SF_TMEM_COL,
                  EPI_THREADS = P::EPI_THREADS, SCALE_WARP0 = P::SCALE_WARP0, EPI_GROUPS = P::EPI_GROUPS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ DivTable2 tab;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *full = bars, *empty = bars + STAGES, *sf_ready = bars + 2 * STAGES, *acc_full = bars + 3 * STAGES,
             *acc_empty = acc_full + ACC_BUFS, *drain = acc_empty + ACC_BUFS, *qa_ready = drain + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Set-up that reads nothing the previous kernel writes runs before the
    // dependency wait, overlapping that kernel's tail: the division table (a
    // kernel parameter), the barriers, the TMEM allocation and the tensor-map
    // prefetch.
    pdl_trigger();
    if (EPI == 0) load_div_table(&tab, tab_in);
    // CTA pairs: rank 0 issues the MMAs; its sf_ready and acc_empty barriers
    // take the arrivals of both CTAs' scale writers and epilogue warps.
    const uint32_t rank = CTA2 ? cluster_rank() : 0u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_ready[s], CTA2 ? 2 * NUM_SCALE_WARPS : NUM_SCALE_WARPS);
        }
        for (int i = 0; i < ACC_BUFS; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], CTA2 ? 2 * P::NUM_EPI_WARPS : EPI_THREADS / EPI_GROUPS);
        }
        mbar_init(drain, 1);
        if (QA) mbar_init(qa_ready, P::NUM_EPI_WARPS);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
        if (DEC) prefetch_tmap(&tmap_a16);
    }
    if (warp == 1) {
        if (CTA2) {
            // one warp of each CTA of the pair, together: the same columns in both
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    // QA, early weights: the CTA's tiles from the call's inputs (no dependency wait)
    const QaRoute *qr = reinterpret_cast<const QaRoute *>(smem + P::OFF_QAR);
    const EarlyRoute *er = reinterpret_cast<const EarlyRoute *>(smem + P::OFF_QAR);
    constexpr bool early = EARLY && !UE;
    if (QA && warp == 2) qa_route(p, reinterpret_cast<QaRoute *>(smem + P::OFF_QAR), lane);
    if (early && warp == 2) early_route(p, reinterpret_cast<EarlyRoute *>(smem + P::OFF_QAR), lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (CTA2) cluster_sync_all();  // the peer's barriers are initialised before any arrival on them

    if (!QA && !early) pdl_wait();  // the previous kernel's outputs (A operand, row maps, status)
    // w2's small-batch plan: the routing's tile map (at most 130 m-tiles) into
    // shared memory beside the header read, one round trip instead of the
    // header's then the tile's expert's
    constexpr bool STE = EPI == 1 && DEC && !EARLY;
    const int *ste = reinterpret_cast<const int *>(smem + P::OFF_QAR);
    int hdr_mtiles = 0, hdr_status = 0;
    if constexpr (STE) {
        hdr_mtiles = p.hdr->num_mtiles;
        hdr_status = p.hdr->status;
        int *ste_w = reinterpret_cast<int *>(smem + P::OFF_QAR);
        const int cap = min(p.mtiles_cap, P::QAR_BYTES / 4);
        for (int j = threadIdx.x; j < cap; j += P::NUM_THREADS) ste_w[j] = p.tile_expert[j];
        __syncthreads();
    }
    constexpr int W = DEC ? 64 : 128;  // w13 tile width in h columns
    const int NT = EPI == 0 ? (p.gate_up_I + W - 1) / W : p.N / 128;
    // w13 pairs: units of two m-tiles; w2: the m-tiles that hold rows
    const int MT = QA      ? (qr->bad ? 0 : qr->mtiles)
                   : early ? (er->bad ? 0 : er->mtiles)
                   : CTA2  ? p.hdr->num_mtiles / 2
                   : (EPI == 1 && p.live_mtiles) ? p.hdr->num_live_mtiles
                   : STE ? hdr_mtiles
                         : p.hdr->num_mtiles;
    const int ntiles = MT * NT;
    const int KT = (p.K + BK - 1) / BK;
    // work is shared out per CTA, or per CTA pair
    const int G = (int)gridDim.x >> (CTA2 ? 1 : 0), b = (int)blockIdx.x >> (CTA2 ? 1 : 0);
    // w2: tile pairs share A when all of a tile's A stages fit the slots, and
    // when pairing (units of two tiles) adds at most 1/32 to the busiest CTA's
    // tile count: with few tiles per CTA, as in decode, that tail costs more
    // than the A loads it saves
    const int per_cta = (ntiles + G - 1) / G, per_cta_paired = 2 * ((MT * (NT / 2) + G - 1) / G);
    const bool paired =
        EPI == 1 && !DEC && KT <= P::A_SLOTS && NT % 2 == 0 && per_cta_paired * 32 <= per_cta * 33;
    const int nunits = paired ? MT * (NT / 2) : ntiles;
    const int n_i = nunits > b ? ((nunits - b + G - 1) / G) * (paired ? 2 : 1) : 0;  // this CTA's tiles
    // QA keeps one m-tile's A for the whole kernel: the host takes it only
    // when no CTA gets a second tile (a broken promise is reported, not run)
    // (and w2's small-batch plan holds at most QAR_BYTES / 4 m-tiles in its copy of the tile map)
    const bool plan_broken = (QA && n_i > 1) || (STE && MT > P::QAR_BYTES / 4);
    if ((!QA && !early && (STE ? hdr_status : p.hdr->status) != 0) || n_i == 0 || plan_broken) {
        // nothing to do (same decision in every thread, and in both CTAs of a
        // pair): give TMEM back.  QA, early weights: after the dependency
        // wait, so that this grid completes after the kernels before it.
        if (QA || early) pdl_wait();
        if (plan_broken && threadIdx.x == 0) atomicOr(&p.hdr->error_flags, kErrPlan);
        if (warp == 1) {
            if (CTA2)
                asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(*tmem_slot),
                             "r"(TMEM_COLS)
                             : "memory");
            else
                asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(*tmem_slot),
                             "r"(TMEM_COLS)
                             : "memory");
        }
        return;
    }

    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t stage = 0, phase = 0;
        uint32_t issued = 0;           // bit s: stage s has had a load issued
        uint32_t last_parity = 0;      // bit s: parity of that last load's phase
        bool ok = true;
        const size_t b_sf_expert = (size_t)(p.N / 128) * p.b_kc * SF_TILE;  // prepared scale bytes per expert
        // Early weights: the first ring stages (all of them, or all the loads
        // when fewer) get their weight loads before the dependency wait and
        // their A loads (the quantiser's output) once it returns.
        bool waited = !early;
        int nd = 0;  // stages loaded so far before the wait (stage s = s, tile 0 .. )
        for (int i = 0; i < n_i && ok; ++i) {
            const TileInfo<EPI> ti = QA      ? qa_tile<EPI>(p, qr)
                                     : early ? early_tile<EPI>(p, er, b + i * G, NT, MT, W)
                                             : seq_tile<EPI, CTA2, STE>(p, i, NT, MT, paired, W, ste);
            const bool fill_a = !paired || (i & 1) == 0;  // w2: the first tile of a pair brings A
            const uint8_t *b_sf = p.b_sf + (size_t)ti.e * b_sf_expert +
                                  (size_t)(EPI == 0 ? 2 * (ti.hc0 >> 7) : ti.nt) * p.b_kc * SF_TILE;
            // w13: hc gate rows and hc up rows (a pair: rank 0 the gate rows, rank 1 the up rows)
            const uint32_t b_bytes = EPI == 0 ? (uint32_t)ti.hc * (CTA2 ? 1 : 2) * (BK / 2) : (uint32_t)B_BYTES;
            const uint32_t sfb_bytes = (uint32_t)ti.nblk * 4 * SF_TILE;
            for (int kt = 0; kt < KT; ++kt) {
                const int kx = kt * (BK / 2);
                // (a pair: released by rank 0's commit to both CTAs)
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                uint64_t *fb = &full[stage];
                const bool a_now = EPI == 0 || fill_a;
                // A: the whole m-tile, or (small-batch plans) its first DEC_ROWS rows
                // (QA: neither A nor its scales, quantised in the kernel)
                const uint32_t a_bytes = DEC ? (uint32_t)(P::DEC_ROWS * BK / 2) : (uint32_t)A_BYTES;
                mbar_expect_tx(fb, QA ? b_bytes + sfb_bytes
                                      : (a_now || DEC ? a_bytes : 0u) + b_bytes + SFA_BYTES + sfb_bytes);
                uint8_t *sb = smem + OFF_B + stage * B_BYTES;
                if (!waited) {
                    ++nd;
                } else if constexpr (QA) {
                } else if constexpr (DEC) {
                    for (int r = 0; r < P::DEC_ROWS; r += 16)
                        tma_2d(smem + OFF_A + stage * P::A_STRIDE + r * (BK / 2), &tmap_a16, kx, ti.mt * BM + r, fb);
                } else if constexpr (EPI == 0) {
                    tma_2d(smem + OFF_A + stage * A_BYTES, &tmap_a, kx, ti.mt * BM, fb);
                } else if (fill_a) {
                    const int f = (paired ? (i >> 1) : i) * KT + kt;  // A fill f goes to slot f % A_SLOTS
                    tma_2d(smem + P::OFF_AS + (f % P::A_SLOTS) * A_BYTES, &tmap_a, kx, ti.mt * BM, fb);
                }
                if (EPI == 0 && CTA2) {
                    // this CTA's half of the B tile: the hc gate rows (rank 0)
                    // or the hc up rows (rank 1), in 64-row boxes
                    const int first = ti.e * 2 * p.gate_up_I + ti.hc0 + (rank ? p.gate_up_I : 0);
                    for (int r = 0; r < ti.hc; r += 64) tma_2d(sb + r * (BK / 2), &tmap_b, kx, first + r, fb);
                } else if (EPI == 0) {
                    // hc gate rows, then the hc matching up rows, in 64-row boxes
                    const int gate = ti.e * 2 * p.gate_up_I + ti.hc0;
                    for (int r = 0; r < ti.hc; r += 64) {
                        tma_2d(sb + r * (BK / 2), &tmap_b, kx, gate + r, fb);
                        tma_2d(sb + (ti.hc + r) * (BK / 2), &tmap_b, kx, gate + p.gate_up_I + r, fb);
                    }
                } else {
                    tma_2d(sb, &tmap_b, kx, ti.e * p.N + ti.nt * 128, fb);
                }
                if (!QA && waited)
                    bulk_g2s(smem + OFF_SFA + stage * SFA_BYTES,
                             p.a_sf + ((size_t)ti.mt * p.a_kc + 4 * kt) * SF_TILE, SFA_BYTES, fb);
                bulk_g2s(smem + OFF_SFB + stage * SFB_BYTES, b_sf + (size_t)4 * kt * ti.nblk * SF_TILE, sfb_bytes,
                         fb);
                issued |= 1u << stage;
                last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (!waited && nd == STAGES) {
                    pdl_wait();
                    waited = true;
                    early_a_loads<EPI, P, DEC>(p, smem, full, &tmap_a, &tmap_a16, nd, b, G, NT, MT, KT);
                }
            }
        }
        if (!waited) {
            pdl_wait();
            early_a_loads<EPI, P, DEC>(p, smem, full, &tmap_a, &tmap_a16, nd, b, G, NT, MT, KT);
        }
        if (!ok) {
            *abort_flag = 1;
            atomicOr(&p.hdr->error_flags, kErrTimeoutProducer);
        }
        // Drain: every issued load has landed before the CTA exits.
        for (int s = 0; s < STAGES; ++s)
            if (issued & (1u << s)) mbar_wait(&full[s], (last_parity >> s) & 1u, nullptr, kDrainLimitNs);
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ------------------------------------------------ MMA issuer
        // (a pair: rank 0 issues the M256 MMAs for both CTAs, waits on barriers
        // both CTAs arrive on, and commits to the barriers of both)
        // The issuing warp shares its scheduler with busy epilogue warps, so
        // the loop is kept short: descriptors advance by constants (a 64-K
        // step is 32 bytes = 2 descriptor units; a stage is a fixed stride)
        // and a full stage's four MMAs are unrolled.
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool ok = true;
        const uint64_t da0 = desc_sw128(su32(smem + (P::A_SLOTS > 0 ? P::OFF_AS : OFF_A))),
                       db0 = desc_sw128(su32(smem + OFF_B));
        const uint32_t sf0 = tmem + SF_TMEM_COL;
        const int k_full = p.K / BK;  // stages with four 64-K steps
        // QA: the A slices are written by the epilogue warps (generic proxy,
        // fenced to the async proxy before their arrival)
        if (QA && !mbar_wait(qa_ready, 0, abort_flag, kWaitLimitNs)) ok = false;

        for (int i = 0; i < n_i && ok; ++i) {
            const int nt = (b + i * G) % NT;  // w13: the tile's width (w2 takes N128 throughout)
            const uint32_t idesc = idesc_for(EPI == 0 ? 2 * min(W, p.gate_up_I - W * nt) : 128, CTA2 ? 2 * BM : BM);
            if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + acc * P::BN;
            for (int kt = 0; kt < KT; ++kt) {
                // the scale writers arrive on sf_ready[stage] only after they
                // have seen the stage's loads land (full[stage])
                if (!mbar_wait(&sf_ready[stage], phase, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // w2: the A fill this stage reads (landed with this tile's, or
                // for the second of a pair the first's, ring stage)
                int sl = QA ? kt : stage;  // QA: the persistent slice of this K step
                if constexpr (P::A_SLOTS > 0) sl = ((paired ? (i >> 1) : i) * KT + kt) % P::A_SLOTS;
                const uint64_t da = da0 + (uint64_t)(sl * (P::A_STRIDE >> 4));
                const uint64_t db = db0 + (uint64_t)(stage * (B_BYTES >> 4));
                const uint32_t sfa = sf0 + stage * SF_COLS, sfb = sfa + 16;
                if constexpr (CTA2) {
                    if (kt < k_full) {
                        tc_mma_pair(d, da, db, idesc, sfa, sfb, kt != 0);
                        tc_mma_pair(d, da + 2, db + 2, idesc, sfa + 4, sfb + SFB_STEP, 1u);
                        tc_mma_pair(d, da + 4, db + 4, idesc, sfa + 8, sfb + 2 * SFB_STEP, 1u);
                        tc_mma_pair(d, da + 6, db + 6, idesc, sfa + 12, sfb + 3 * SFB_STEP, 1u);
                    } else {
                        const int ksteps = (p.K - kt * BK) / 64;
                        for (int j = 0; j < ksteps; ++j)
                            tc_mma_pair(d, da + 2 * j, db + 2 * j, idesc, sfa + 4 * j, sfb + SFB_STEP * j,
                                        (kt | j) != 0);
                    }
                    tc_commit_pair(&empty[stage]);
                } else {
                    if (kt < k_full) {
                        tc_mma(d, da, db, idesc, sfa, sfb, kt != 0);
                        tc_mma(d, da + 2, db + 2, idesc, sfa + 4, sfb + SFB_STEP, 1u);
                        tc_mma(d, da + 4, db + 4, idesc, sfa + 8, sfb + 2 * SFB_STEP, 1u);
                        tc_mma(d, da + 6, db + 6, idesc, sfa + 12, sfb + 3 * SFB_STEP, 1u);
                    } else {
                        const int ksteps = (p.K - kt * BK) / 64;
                        for (int j = 0; j < ksteps; ++j)
                            tc_mma(d, da + 2 * j, db + 2 * j, idesc, sfa + 4 * j, sfb + SFB_STEP * j, (kt | j) != 0);
                    }
                    tc_commit(&empty[stage]);
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (CTA2)
                tc_commit_pair(&acc_full[acc]);
            else
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
        // Drain: all issued tcgen05 work completes before TMEM is released
        // (a pair: both CTAs wait for it below, before either releases its
        // tensor memory or shared memory).
        if (CTA2) {
            tc_commit_pair(drain);
        } else {
            tc_commit(drain);
            mbar_wait(drain, 0, nullptr, kDrainLimitNs);
        }
    } else if (warp >= SCALE_WARP0) {
        // ------------------------------------------------ scale writers
        // Each warp owns one TMEM lane quarter and writes the stage's scales
        // there with tcgen05.st: per 64-K step and 128-row block, the 16 bytes
        // of row (lane) of the 128x4-scale tile (the scales of rows lane,
        // lane+32, lane+64, lane+96) go to four consecutive columns of every
        // lane quarter, the layout the block-scaled MMA reads.  With N256 the
        // second 128-row block of B follows the first at +4 columns.  Register
        // stores from four warps in parallel keep the MMA issuer free of the
        // smem -> TMEM copy queue.  A stage's slot is rewritten only after the
        // producer has refilled the stage, i.e. after the MMAs that read it
        // have finished.
        const int quarter = warp & 3;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        // UE8M0: word q of this lane's 16 bytes holds row q * 32 + lane of
        // the m-tile; its bytes are carried with that row's shift.  The rows'
        // largest bytes are loaded one tile ahead, off the stage's path.
        int rmax_next[4] = {0, 0, 0, 0};
        if (QA && !mbar_wait(qa_ready, 0, abort_flag, kWaitLimitNs)) ok = false;  // the A scale tiles
        if (UE && n_i > 0) {
            const int mt0 = seq_tile<EPI, CTA2>(p, 0, NT, MT, paired, W).mt;
#pragma unroll
            for (int q = 0; q < 4; ++q) rmax_next[q] = __ldg(p.a_row_max + mt0 * BM + q * 32 + lane);
        }
        for (int i = 0; i < n_i && ok; ++i) {
            const TileInfo<EPI> ti = QA      ? qa_tile<EPI>(p, qr)
                                     : early ? early_tile<EPI>(p, er, b + i * G, NT, MT, W)
                                             : seq_tile<EPI, CTA2, STE>(p, i, NT, MT, paired, W, ste);
            uint32_t c4[4] = {0u, 0u, 0u, 0u};
            if (UE) {
#pragma unroll
                for (int q = 0; q < 4; ++q) c4[q] = ue8m0_row_shift((uint32_t)rmax_next[q]) * 0x01010101u;
                if (i + 1 < n_i) {
                    const int mt1 = seq_tile<EPI, CTA2>(p, i + 1, NT, MT, paired, W).mt;
#pragma unroll
                    for (int q = 0; q < 4; ++q) rmax_next[q] = __ldg(p.a_row_max + mt1 * BM + q * 32 + lane);
                }
            }
            for (int kt = 0; kt < KT; ++kt) {
                if (!mbar_wait(&full[stage], phase, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                const uint32_t sfa_t = tmem + lane_off + SF_TMEM_COL + stage * SF_COLS, sfb_t = sfa_t + 16;
                const uint4 *ssfa =
                    reinterpret_cast<const uint4 *>(smem + OFF_SFA + (QA ? kt : (int)stage) * SFA_BYTES) + lane;
                const uint4 *ssfb = reinterpret_cast<const uint4 *>(smem + OFF_SFB + stage * SFB_BYTES) + lane;
                uint4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = ssfa[32 * j];
                if (UE) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        v[j] = make_uint4(ue8m0_carried4(v[j].x, c4[0]), ue8m0_carried4(v[j].y, c4[1]),
                                          ue8m0_carried4(v[j].z, c4[2]), ue8m0_carried4(v[j].w, c4[3]));
                }
                tmem_st16(sfa_t, v);
                if (DEC) {
                    // 64-column tiles, four columns per 64-K step: the tile's
                    // 64 gate rows are words 2c, 2c+1 of the gate tile's 16
                    // bytes (rows 64c + lane, 64c + 32 + lane), its 64 up rows
                    // the same words of the up tile; a native 64 + 64 tile as is
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (ti.compose) {
                            const uint4 g = ssfb[32 * (2 * j)], u = ssfb[32 * (2 * j + 1)];
                            v[j] = ti.compose == 1 ? make_uint4(g.x, g.y, u.x, u.y) : make_uint4(g.z, g.w, u.z, u.w);
                        } else {
                            v[j] = ssfb[32 * j];
                        }
                    }
                    tmem_st16(sfb_t, v);
                } else if (SFB_STEP == 4) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[j] = ssfb[32 * j];
                    tmem_st16(sfb_t, v);
                } else {
                    // column 4i holds tile i of the stage: (step i/2, block i%2)
                    // for a full tile; a narrow tile has one block per step
                    // and leaves the odd slots as copies.
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int i = 4 * h + j;
                            v[j] = ti.nblk == 2 ? ssfb[32 * i] : ssfb[32 * (i >> 1)];
                        }
                        tmem_st16(sfb_t + 16 * h, v);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (CTA2)
                        mbar_arrive_rank0(&sf_ready[stage]);  // both CTAs' scales feed rank 0's MMA
                    else
                        mbar_arrive(&sf_ready[stage]);
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(&p.hdr->error_flags, kErrTimeoutMma);
        }
    } else if (warp >= 2 && warp < SCALE_WARP0) {
        // ------------------------------------------------ epilogue
        const int ew = warp - 2;                         // 0 .. epilogue warps - 1
        const int group = ew / (P::NUM_EPI_WARPS / EPI_GROUPS);  // w2: tiles of this group's parity
        const int quarter = warp & 3;                    // TMEM lanes this warp may read
        const int half = (ew >> 2) & 1;                  // w2: which half of the tile's columns it owns
        const int part = ew >> 2;                        // w13: which slice of the tile's h columns
        const int r_in = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        float *xp = reinterpret_cast<float *>(smem + OFF_XPOSE) + ew * 32 * XPOSE_LD;
        const uint32_t acc = EPI_GROUPS == 2 ? (uint32_t)group : 0u;
        uint32_t acc_phase = 0;
        bool ok = true;
        // w13: the FP32 output is cleared for the w2 kernel's reductions, a
        // slice after each tile, so that the stores use the HBM bandwidth the
        // GEMM leaves idle instead of delaying the first accumulator.  Each
        // active CTA owns a contiguous range of it.
        long long z_next = 0, z_end = 0, z_slice = 0;
        float4 *z4 = reinterpret_cast<float4 *>(p.zero_out);
        if (EPI == 0 && p.zero_out) {
            const long long n4 = p.zero_floats >> 2;
            const long long active = min((long long)gridDim.x, (long long)ntiles << (CTA2 ? 1 : 0));
            const long long per_cta = (n4 + active - 1) / active;
            const long long my_tiles = n_i;
            z_next = min(n4, (long long)blockIdx.x * per_cta);
            z_end = min(n4, z_next + per_cta);
            z_slice = (per_cta + my_tiles - 1) / my_tiles;
        }
        int n_epi = n_i;  // tiles whose results this CTA writes
        float qa_g2 = 1.0f, qa_alpha = 1.0f;  // QA: the expert's a2 scale and alpha
        if (early) {
            // the routing's tile map, the quantiser's A and the status from here
            pdl_wait();
            if (p.hdr->status != 0) n_epi = 0;
        }
        if constexpr (QA) {
            // The m-tile's live rows quantised into the persistent A slices,
            // one 16-element block per thread and item, by the a1 quantiser's
            // block routine, at the bytes a 128-byte-swizzled TMA load of
            // 16-row boxes would fill; their scale bytes into the persistent
            // scale tiles.  x is an input of the call: it was complete before
            // this kernel could start (the routing kernel lets it start only
            // after its own dependency wait).
            // (the expert's scales are the scale check's reciprocals and
            // alpha, by the same operations; loaded with the first x rows)
            const int nlive = qr->nlive, nblk = p.K >> 4, eq = max(qr->e, 0);
            const float in1 = ld_cg(p.in_scale1 + eq), in2 = ld_cg(p.in_scale2 + eq), ws2 = ld_cg(p.w13_scale2 + eq);
            const float g = __frcp_rn(in1);
            qa_g2 = __frcp_rn(in2);
            qa_alpha = __frcp_rn(__fmul_rn(g, __frcp_rn(ws2)));
            for (int it = ew * 32 + lane; it < nlive * nblk; it += EPI_THREADS) {
                const int r = it / nblk, kb = it - r * nblk;
                const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (size_t)(qr->f[r] / p.k) * p.K + kb * 16);
                const uint4 v0 = ld_cg(src), v1 = ld_cg(src + 1);
                const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                f32x2 xv[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) xv[j] = bf16x2_to_f32x2(wv[j]);
                uint32_t sb;
                const uint2 q = quant_block16(xv, amax16_bf16(wv), g, &tab, sb);
                const int kt = kb >> 4, kb16 = kb & 15;
                *reinterpret_cast<uint2 *>(smem + OFF_A + kt * P::A_STRIDE + r * (BK / 2) +
                                           (((kb16 >> 1) ^ (r & 7)) << 4) + ((kb16 & 1) << 3)) = q;
                smem[OFF_SFA + kt * SFA_BYTES + (kb16 >> 2) * SF_TILE + (r & 31) * 16 + (r >> 5) * 4 + (kb16 & 3)] =
                    (uint8_t)sb;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // for the MMAs' reads
            __syncwarp();
            if (lane == 0) mbar_arrive(qa_ready);
            // Writes only from here: after the scale check and routing, and
            // only when they passed.  The m-tile's first tile (one CTA per
            // m-tile) copies its A rows to the workspace's A operand.
            pdl_wait();
            if (p.hdr->status != 0) n_epi = 0;
            if (n_epi > 0 && qr->nt == 0) {
                const int row0 = qr->mt * BM;
                uint8_t *const aq = const_cast<uint8_t *>(p.a_q);
                uint8_t *const asf = const_cast<uint8_t *>(p.a_sf);
                for (int it = ew * 32 + lane; it < nlive * nblk; it += EPI_THREADS) {
                    const int r = it / nblk, kb = it - r * nblk, row = row0 + r;
                    const int kt = kb >> 4, kb16 = kb & 15;
                    *reinterpret_cast<uint2 *>(aq + (size_t)row * (p.K >> 1) + kb * 8) =
                        *reinterpret_cast<const uint2 *>(smem + OFF_A + kt * P::A_STRIDE + r * (BK / 2) +
                                                         (((kb16 >> 1) ^ (r & 7)) << 4) + ((kb16 & 1) << 3));
                    asf[((size_t)(row >> 7) * p.a_kc + (kb >> 2)) * SF_TILE + (row & 31) * 16 + ((row >> 5) & 3) * 4 +
                        (kb & 3)] = smem[OFF_SFA + kt * SFA_BYTES + (kb16 >> 2) * SF_TILE + (r & 31) * 16 +
                                         (r >> 5) * 4 + (kb16 & 3)];
                }
            }
        }
        for (int i = group; i < n_epi; i += EPI_GROUPS) {
            // everything the tile needs besides the accumulator is fetched
            // before waiting for it
            const TileInfo<EPI> ti = QA ? qa_tile<EPI>(p, qr) : seq_tile<EPI, CTA2, STE>(p, i, NT, MT, paired, W, ste);
            const int e = ti.e, nt = ti.nt;
            const int row = ti.mt * BM + r_in;
            bool valid;
            float s0, s1;  // w13: alpha, g2; w2: routing weight * alpha2
            int t = 0;     // w2: token of the row
            if (QA) {
                valid = r_in < qr->nlive;
                s0 = qa_alpha;
                s1 = qa_g2;
            } else if (EPI == 0) {
                valid = row < p.pad_off[e] + p.counts[e];
                s0 = p.alpha[e];
                s1 = p.g2[e];
            } else {
                const int f = p.row_src[row];  // -1 on padding rows
                valid = f >= 0;
                s0 = valid ? __fmul_rn(p.topk_w[f], p.alpha[e]) : 0.0f;
                s1 = 0.0f;
                t = valid ? f / p.k : 0;
            }
            // UE8M0: the A row's carried scales take 2^(shift - 120) back (an
            // exact product), and the weight rows' factors are applied per
            // column.  Those are loaded here, before the accumulator wait, one
            // column per lane: w13 lane l holds the gate and up factors of
            // columns l and 32 + l of this warp's slice, w2 the four columns
            // it reduces in each 32-column chunk.
            float4 colf[2] = {make_float4(1.f, 1.f, 1.f, 1.f), make_float4(1.f, 1.f, 1.f, 1.f)};
            if (UE) {
                s0 *= ue8m0_row_factor(ue8m0_row_shift((uint32_t)p.a_row_max[row]));
                if (EPI == 0) {
                    const int w0 = part * (ti.hc / (P::NUM_EPI_WARPS / 4));
                    const float *fg = p.b_row_factor + (size_t)e * p.N + ti.hc0 + w0;
                    const int hw = ti.hc / (P::NUM_EPI_WARPS / 4);
                    colf[0].x = fg[lane];
                    colf[0].y = fg[p.gate_up_I + lane];
                    colf[0].z = hw > 32 ? fg[32 + lane] : 1.f;
                    colf[0].w = hw > 32 ? fg[p.gate_up_I + 32 + lane] : 1.f;
                } else {
                    const float *fc = p.b_row_factor + (size_t)e * p.N + nt * 128 + (lane & 7) * 4;
                    colf[0] = __ldg(reinterpret_cast<const float4 *>(fc + 64 * half));
                    colf[1] = __ldg(reinterpret_cast<const float4 *>(fc + 64 * half + 32));
                }
            }
            if (!mbar_wait(&acc_full[acc], acc_phase, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t col0 = lane_base + acc * P::BN;
            if (EPI == 0) {
                // This warp's h columns: [w0, w0 + hw) of the tile, hw = hc/2,
                // w0 = half * hw; gate accumulator columns w0.., up columns
                // hc + w0...  h = SiLU(alpha * gate) * (alpha * up) is formed
                // 32 columns at a time and the accumulator released once all
                // of it is in registers.
                const float alpha = s0, g2 = s1;
                const f32x2 aa = pack_f32x2(alpha, alpha);
                const int hw = ti.hc / (P::NUM_EPI_WARPS / 4), w0 = part * hw;
                const int nblocks = hw >> 4;  // blocks of 16 of this warp
                f32x2 h[4][8];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (c * 32 >= hw) break;
                    float gate[32], up[32];
                    tmem_ld16(col0 + w0 + 32 * c, gate);
                    tmem_ld16(col0 + w0 + 32 * c + 16, gate + 16);
                    tmem_ld16(col0 + ti.hc + w0 + 32 * c, up);
                    tmem_ld16(col0 + ti.hc + w0 + 32 * c + 16, up + 16);
                    tmem_wait_ld(gate, up);
                    if (32 * (c + 1) >= hw) {
                        // the whole accumulator slice is in registers (a pair:
                        // one arrival per warp, on rank 0's barrier)
                        tc_fence_before();
                        if (CTA2) {
                            __syncwarp();
                            if (lane == 0) mbar_arrive_rank0(&acc_empty[acc]);
                        } else {
                            mbar_arrive(&acc_empty[acc]);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        f32x2 gs = mul_f32x2(pack_f32x2(gate[2 * i], gate[2 * i + 1]), aa);
                        f32x2 us = mul_f32x2(pack_f32x2(up[2 * i], up[2 * i + 1]), aa);
                        if (UE) {
                            const float fg = c == 0 ? colf[0].x : colf[0].z, fu = c == 0 ? colf[0].y : colf[0].w;
                            gs = mul_f32x2(gs, pack_f32x2(__shfl_sync(0xffffffffu, fg, 2 * i),
                                                          __shfl_sync(0xffffffffu, fg, 2 * i + 1)));
                            us = mul_f32x2(us, pack_f32x2(__shfl_sync(0xffffffffu, fu, 2 * i),
                                                          __shfl_sync(0xffffffffu, fu, 2 * i + 1)));
                        }
                        h[2 * c + (i >> 3)][i & 7] = mul_f32x2(pack_f32x2(silu(lo_f32(gs)), silu(hi_f32(gs))), us);
                    }
                }
                uint32_t sfw = 0, sf_max = 0;
                const int hcol_tile = ti.hc0 + w0;  // first h column of this warp
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    if (b >= nblocks) break;
                    float amax = 0.0f;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        amax = fmaxf(amax, fmaxf(fabsf(lo_f32(h[b][i])), fabsf(hi_f32(h[b][i]))));
                    const int hcol = hcol_tile + 16 * b;
                    if (p.h_dump && valid) {
                        float4 *hd = reinterpret_cast<float4 *>(p.h_dump + (size_t)row * p.I + hcol);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            hd[i] = make_float4(lo_f32(h[b][2 * i]), hi_f32(h[b][2 * i]), lo_f32(h[b][2 * i + 1]),
                                                hi_f32(h[b][2 * i + 1]));
                    }
                    uint32_t sb;
                    uint2 pk;
                    if (UE) {
                        pk = quant_block16_ue8m0(h[b], amax, g2, sb);
                        sf_max = max(sf_max, sb);
                    } else {
                        pk = quant_block16(h[b], amax, g2, &tab, sb);
                    }
                    if (valid) *reinterpret_cast<uint2 *>(p.a2q + (size_t)row * (p.I >> 1) + (hcol >> 1)) = pk;
                    sfw |= sb << (8 * b);
                }
                if (valid) {
                    // four scales = one 64-column chunk (full tile), or two =
                    // half a chunk (narrow tile)
                    uint8_t *sfp = p.sf2 + swz_sf_offset(row, hcol_tile >> 6, p.kc2) + ((hcol_tile & 63) >> 4);
                    if (nblocks == 4)
                        *reinterpret_cast<uint32_t *>(sfp) = sfw;
                    else if (nblocks == 2)
                        *reinterpret_cast<uint16_t *>(sfp) = (uint16_t)sfw;
                    else
                        *sfp = (uint8_t)sfw;
                    if (nt == NT - 1 && part == 0)
                        for (int cc = p.I >> 6; cc < p.kc2; ++cc)
                            *reinterpret_cast<uint32_t *>(p.sf2 + swz_sf_offset(row, cc, p.kc2)) = 0u;
                    if (UE) atomicMax(p.out_row_max + row, (int)sf_max);  // the w2 kernel carries a2 by it
                }
            } else {
                // out[t, cols] += w[t, j] * alpha2 * y2 on this warp's 64 columns,
                // 32 at a time, transposed through shared memory so that each
                // reduction instruction covers four contiguous 128-byte row
                // segments.
                const float scale = s0;
                const int sub = lane >> 3, cc = (lane & 7) * 4;
                if (DEC) {
                    // a tile holds one or two live rows: each valid lane adds
                    // its own row's 32 columns, from registers
#pragma unroll 1
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const int cbase = 64 * half + 32 * c2;
                        float v[32];
                        tmem_ld16(col0 + cbase, v);
                        tmem_ld16(col0 + cbase + 16, v + 16);
                        tmem_wait_ld(v);
                        if (c2 == 1) {
                            tc_fence_before();
                            mbar_arrive(&acc_empty[acc]);
                        }
                        if (valid) {
                            float *o = p.out + (size_t)t * p.H + nt * 128 + cbase;
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                red_add_v4(o + 4 * j, v[4 * j] * scale, v[4 * j + 1] * scale, v[4 * j + 2] * scale,
                                           v[4 * j + 3] * scale);
                        }
                    }
                }
#pragma unroll 1
                for (int c2 = 0; c2 < (DEC ? 0 : 2); ++c2) {
                    const int cbase = 64 * half + 32 * c2;
                    float v[32];
                    tmem_ld16(col0 + cbase, v);
                    tmem_ld16(col0 + cbase + 16, v + 16);
                    tmem_wait_ld(v);
                    if (c2 == 1) {
                        tc_fence_before();
                        mbar_arrive(&acc_empty[acc]);
                    }
                    float4 *xrow = reinterpret_cast<float4 *>(xp + lane * XPOSE_LD);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        xrow[j ^ (lane & 7)] = make_float4(v[4 * j] * scale, v[4 * j + 1] * scale,
                                                           v[4 * j + 2] * scale, v[4 * j + 3] * scale);
                    __syncwarp();
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int rr = it * 4 + sub;
                        const int t_r = __shfl_sync(0xffffffffu, t, rr);
                        const int ok_r = __shfl_sync(0xffffffffu, (int)valid, rr);
                        float4 src = reinterpret_cast<const float4 *>(xp + rr * XPOSE_LD)[(lane & 7) ^ (rr & 7)];
                        if (UE) {  // the weight rows' factors of this lane's four columns (exact products)
                            const float4 f = c2 == 0 ? colf[0] : colf[1];
                            src = make_float4(src.x * f.x, src.y * f.y, src.z * f.z, src.w * f.w);
                        }
                        if (ok_r)
                            red_add_v4(p.out + (size_t)t_r * p.H + nt * 128 + cbase + cc, src.x, src.y, src.z,
                                       src.w);
                    }
                    __syncwarp();
                }
            }
            if (EPI == 0 && z_next < z_end) {
                const long long stop = min(z_end, z_next + z_slice);
                for (long long i = z_next + (threadIdx.x - 64); i < stop; i += EPI_THREADS)
                    z4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                z_next = stop;
            }
            acc_phase ^= 1u;  // each group owns one accumulator
        }
        if (!ok) {
            *abort_flag = 1;
            atomicOr(&p.hdr->error_flags, kErrTimeoutEpilogue);
        }
    }
    // a pair: every MMA rank 0 issued has completed (they read both CTAs'
    // shared and tensor memory) before either CTA releases anything
    if (CTA2 && warp == 1 && lane == 0) mbar_wait(drain, 0, nullptr, kDrainLimitNs);
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if (CTA2)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                         : "memory");
    }
}

// ---------------------------------------------------------------- host side
// 2-D byte tensor [rows, row_bytes] with a (128 bytes x box_rows) box, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows)
{
    return make_tensor_map_2d(m, base, row_bytes, rows, 128, box_rows, true);
}

template <int EPI, bool UE, bool CTA2, bool DEC = false, bool QA = false, bool EARLY = false>
cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t st)
{
    using P = Plan<EPI, CTA2, DEC, QA, EARLY>;
    auto kernel = moe_gemm_kernel<EPI, UE, CTA2, DEC, QA, EARLY>;
    // function attributes and the pair form's resident cluster count are per
    // device: taken once on each
    static bool attr_set[64] = {false};
    static int clusters[64] = {0};
    int dev = 0;
    cudaError_t aerr = cudaGetDevice(&dev);
    if (aerr != cudaSuccess) return aerr;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        aerr = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P::SMEM_BYTES);
        if (aerr != cudaSuccess) return aerr;
        if (CTA2) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(2 * (sm_count() / 2));
            q.blockDim = dim3(P::NUM_THREADS);
            q.dynamicSmemBytes = P::SMEM_BYTES;
            cudaLaunchAttribute ca[1];
            ca[0].id = cudaLaunchAttributeClusterDimension;
            ca[0].val.clusterDim.x = 2;
            ca[0].val.clusterDim.y = 1;
            ca[0].val.clusterDim.z = 1;
            q.attrs = ca;
            q.numAttrs = 1;
            int n = 0;
            aerr = cudaOccupancyMaxActiveClusters(&n, kernel, &q);
            if (aerr != cudaSuccess) return aerr;
            if (n < 1) return cudaErrorInvalidConfiguration;
            clusters[dev] = n;
        }
        attr_set[dev] = true;
    }
    CUtensorMap ma, mb, ma16;  // ma16: A in 16-row boxes (the small-batch plan)
    const uint64_t kbytes = (uint64_t)a.K / 2;
    if (!make_map(&ma, a.a_q, kbytes, (uint64_t)a.rows_cap, 128)) return cudaErrorInvalidValue;
    if (!make_map(&ma16, a.a_q, kbytes, (uint64_t)a.rows_cap, 16)) return cudaErrorInvalidValue;
    const uint64_t brows = (uint64_t)a.E * (uint64_t)a.N;
    if (!make_map(&mb, a.b_q, kbytes, brows, a.gate_up_I > 0 ? 64 : 128)) return cudaErrorInvalidValue;
    const long long nt = EPI == 0 ? (a.gate_up_I + (DEC ? 63 : 127)) / (DEC ? 64 : 128) : a.N / 128;
    cudaError_t err;
    if (CTA2) {
        // one resident cluster of two CTAs per SM pair; units are m-tile pairs
        const long long units = (long long)(a.mtiles_cap / 2) * nt;
        int nc = clusters[dev];
        if (units < nc) nc = (int)(units > 0 ? units : 1);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * nc);
        cfg.blockDim = dim3(P::NUM_THREADS);
        cfg.dynamicSmemBytes = P::SMEM_BYTES;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        err = cudaLaunchKernelEx(&cfg, kernel, ma, mb, ma16, a, div_table());
    } else {
        const long long tiles = (long long)a.mtiles_cap * nt;
        int grid = sm_count();
        if (tiles < grid) grid = (int)(tiles > 0 ? tiles : 1);
        err = launch_pdl(kernel, dim3(grid), dim3(P::NUM_THREADS), P::SMEM_BYTES, st, ma, mb, ma16, a, div_table());
    }
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn query_encode_fn()
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
}

static EncodeTiledFn encode_fn()
{
    static const EncodeTiledFn fn = query_encode_fn();  // initialised once, thread-safe
    return fn;
}

bool make_tensor_map_2d(CUtensorMap *m, const void *base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
                        uint32_t box_rows, bool swizzle128)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_bytes, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d) for a %llu x %llu byte tensor", (int)r,
                  (unsigned long long)rows, (unsigned long long)row_bytes);
        return false;
    }
    return true;
}

cudaError_t launch_gemm_w13(const GemmArgs &a, cudaStream_t st)
{
    if (a.pairs) return a.ue8m0 ? launch_gemm<0, true, true>(a, st) : launch_gemm<0, false, true>(a, st);
    if (a.small && !a.ue8m0) {
        if (a.early) return cudaErrorInvalidValue;  // the wide tiles only
        return a.a_inline ? launch_gemm<0, false, false, true, true>(a, st) : launch_gemm<0, false, false, true>(a, st);
    }
    if (a.a_inline) return cudaErrorInvalidValue;  // A is quantised in the kernel by the small-batch plan only
    if (a.early) return a.ue8m0 ? cudaErrorInvalidValue : launch_gemm<0, false, false, false, false, true>(a, st);
    return a.ue8m0 ? launch_gemm<0, true, false>(a, st) : launch_gemm<0, false, false>(a, st);
}
cudaError_t launch_gemm_w2(const GemmArgs &a, cudaStream_t st)
{
    if (a.small && !a.ue8m0)
        return a.early ? launch_gemm<1, false, false, true, false, true>(a, st) : launch_gemm<1, false, false, true>(a, st);
    if (a.early) return cudaErrorInvalidValue;  // the small-batch plan only
    return a.ue8m0 ? launch_gemm<1, true, false>(a, st) : launch_gemm<1, false, false>(a, st);
}

}  // namespace nvfp4
