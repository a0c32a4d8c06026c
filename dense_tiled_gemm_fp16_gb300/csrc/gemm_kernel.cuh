// Persistent, warp-specialised fp16 GEMM for sm_103a: C = A * B with fp16
// operands, fp32 accumulation in tensor memory (TMEM) and fp16 output.
//
// One CTA (or CTA cluster) per SM (pair) walks a list of work units.  A unit
// is a whole output tile, a narrower piece of a tile of the last partial wave
// (tail split along N), or a K segment of a tile (classic split-K, or the
// stream-K tail).  The kernel template gemm_f16_persistent<kPair, kMulti,
// kEpi> has two forms:
//
//   single (kPair = false)  a 128 x BN tile per CTA, cta_group::1 MMAs.  Any
//                           operand layout (TMA or gather), any unit kind.
//   pair   (kPair = true)   clusters of two CTAs; a 256 x BN tile per pair,
//                           one cta_group::2 MMA stream issued by the leader
//                           (rank 0).  Each CTA loads its own 128 rows of A
//                           and its own BN/2 columns of B into its own shared
//                           memory (no multicast), so a CTA moves 2/3 of the
//                           single form's operand bytes per MMA cycle and
//                           fits deeper pipelines.  TMA operands only.
//
// kMulti adds the geometry of batched and grouped launches (per-unit problem,
// trailing batch coordinate of the TMA maps, group row limits); kEpi adds the
// fused output stage (bias, activation, gate/up product).
//
// Roles (8 warps; 256 threads leave each thread up to 255 registers):
//   warps 0-2  producers.  Operands that TMA can address are loaded by one
//              thread with cp.async.bulk.tensor into 128-byte-swizzled shared
//              memory (out-of-range box elements arrive as zeros).  Operands
//              TMA cannot address (unaligned base or pitch, non-unit inner
//              stride) and that the host did not copy to an aligned buffer are
//              gathered by all 96 threads with bounds-checked loads, written in
//              the same swizzled layout and published to the tensor core with
//              fence.proxy.async.  Either way the K tail is zero-filled: an
//              index past K is never wrapped back into range.
//   warp 3     TMEM allocation and the MMA issuer (one thread): 4 x
//              tcgen05.mma (K = 16 each) per 64-wide K block, two K blocks per
//              barrier phase, into one of two TMEM accumulators, so the
//              epilogue of a tile overlaps the main loop of the next.
//   warps 4-7  epilogue.  tcgen05.ld of the fp32 accumulator (warp w reads
//              TMEM lanes 32*(w%4)..+31), the fused stage if any, convert to
//              fp16, then stage 32 x 64 boxes in swizzled shared memory and
//              either TMA-store them (clipped to M x N) or, where TMA cannot
//              store C, write them row by row; the swapped form's transposed C
//              takes per-element bounds-checked stores.  A unit that is a K
//              segment leaves an fp32 partial in the workspace, and the last
//              unit of its tile to finish adds all partials in K order
//              (deterministic) before the store.
//
// Stages form a ring guarded by full/empty mbarriers; accumulators by
// tmem_full/tmem_empty mbarriers.  All waits are bounded (see ptx.cuh).
//
// The decomposition follows the pages' blocked GEMM: each output element has
// exactly one owner and its K reduction is completed before the single store
// ("Triton GEMM: from one output tile to addresses, boundaries and data reuse",
// sections on output ownership and on non-divisible dimensions); the staged,
// multi-buffered K loop is the TileLang tutorial's rung 3 (ch. 14, section 2.3)
// and the double-buffer protocol of the AI-infra page (section 06); split-K
// with a wide accumulator is section 4.1 of the TileLang chapter.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace gemm_f16_dev {

constexpr int kBM = 128;                 // rows per CTA = UMMA M of the single form
constexpr int kBK = 64;                  // K per stage: one 128-byte swizzle row of fp16
constexpr int kMaxStages = 16;
// K blocks (shared-memory slots of 64 K) per pipeline barrier phase: the MMA
// issuer waits once and commits once per kSlots * 4 MMAs, which halves the
// per-K-block cost of the barrier round trip (it cannot overlap the issue).
constexpr int kSlots = 2;
constexpr int kMaxGroups = 64;   // groups of one grouped launch (GEMM_F16_MAX_GROUPS)
constexpr int kNumThreads = 256;         // 8 warps
constexpr int kProducerThreads = 96;     // warps 0-2
constexpr int kEpiWarp0 = 4;
constexpr int kMmaWarp = 3;
// Threads that wait on barriers for long stretches sit on SM sub-partitions
// other than the MMA issuer's (warp 3, sub-partition 3, shared only with the
// epilogue warp 7): the TMA-issuing producer thread is lane 0 of warp 1 (when
// no operand is gathered) and the epilogue thread that waits for accumulators
// is lane 0 of warp 5.
constexpr int kTmaThread = 32;
constexpr int kEpiLead = (kEpiWarp0 + 1) * 32;
constexpr uint32_t kTmemCols = 512;      // two accumulators of up to 256 columns
constexpr uint32_t kAccStride = 256;
constexpr uint32_t kStageABytes = kBM * kBK * 2;        // 16 KiB
constexpr uint32_t kEpiBufBytes = 32 * 64 * 2;           // one warp's 32 x 64 fp16 box
constexpr uint32_t kEpiBytes = 4 * 2 * kEpiBufBytes;     // 4 warps, double-buffered
constexpr uint32_t kBarrierBytes = 512;
constexpr int kStatusTimeout = 6;
constexpr int kStatusBounds = 7;   // debug bounds check: an access was skipped (GEMM_F16_ERR_BOUNDS)
// Spans of the debug bounds check (KernelParams::span_lo / span_hi).
enum : int { kSpanA = 0, kSpanB = 1, kSpanBu = 2, kSpanC = 3 };

// Operand flags.  kOpBox3d: an MN-major TMA operand whose MN extent is a
// multiple of 64 is described as a 3-D tensor (64 MN elements, K, MN / 64
// swizzle-atom columns), so that one copy brings every atom column of a stage
// instead of one copy per 64-wide column.
enum : uint32_t { kOpTma = 1u, kOpMnMajor = 2u, kOpBox3d = 4u };

struct KernelParams {
    CUtensorMap tmA;   // A' (K-major: dims {K, M}; MN-major: dims {M, K})
    CUtensorMap tmB;   // B' (K-major: dims {K, N}; MN-major: dims {N, K})
    CUtensorMap tmB2;  // B' with the box of a tail piece (tail_split > 1): as narrow as the piece
    CUtensorMap tmC;   // C  (dims {N, M}, box 64 x 32): one epilogue warp's rows
    CUtensorMap tmC4;  // C  with a box of 64 x 128: the four epilogue warps' rows in one store
    CUtensorMap tmBu;  // gated fused stage: the up projection's B' (the geometry of tmB)
    // A' and B' with the 64-wide K block as an outer dimension (k2 != 0): one
    // copy brings an operand's boxes of both K blocks of a barrier phase into
    // its two consecutive slots (K-major: dims {64 K, MN, K blocks}; MN-major:
    // {64 MN, 64 K, atom columns, K blocks}; a trailing batch dimension as in
    // tmA / tmB).  Only whole K blocks (kfull = K / 64) are addressed.  The
    // gate/up pair form's rank 1 reads the up projection through tmBu2k.
    CUtensorMap tmA2k;
    CUtensorMap tmB2k;
    CUtensorMap tmBu2k;
    uint32_t k2;
    int kfull;
    const __half* A;   // A'[m,k] = A[m*a_sm + k*a_sk]
    int64_t a_sm, a_sk;
    const __half* B;   // B'[k,n] = B[k*b_sk + n*b_sn]
    int64_t b_sk, b_sn;
    __half* C;         // C'[m,n] = C[m*c_sm + n*c_sn]
    int64_t c_sm, c_sn;
    int64_t M, N, K;
    float* ws;         // split-K partials: [unit][column][row] fp32
    int* counters;     // split-K arrival counters, one per tile, kept at zero between calls
    int* status;       // device status word (kStatusTimeout on a bounded-wait expiry)
    uint64_t timeout_ns;
    int tiles_m, tiles_n, splits, kblocks, num_units, panel, BN, stages;
    uint32_t a_flags, b_flags, c_tma, idesc, tx_bytes, stage_b_bytes, full_count;
    // C that TMA cannot store (unaligned base or pitch, N not a multiple of 8)
    // but with a unit column stride: boxes are staged in shared memory as for
    // TMA and written row by row by the warp (stores of contiguous columns).
    uint32_t c_stage;
    // Debug bounds check (0 off): byte ranges [span_lo, span_hi) of the kernel
    // views A', B', the up projection and C; every gathered load and every
    // per-thread store of C is checked against its range, and one that would
    // leave it is skipped and reported (kStatusBounds).
    uint32_t debug_bounds;
    uintptr_t span_lo[4], span_hi[4];
    // Failure-detection test: the MMA issuer first waits on a barrier that
    // nothing arrives on, so the bounded wait runs out, the CTA aborts and the
    // status word reports the timeout (the host reads it; the context stays
    // usable).  0 in every ordinary call.
    uint32_t test_stall;
    uint32_t epi_smem;   // 1: reserve the 32 KB epilogue buffer (TMA-store staging, fixup landing zone)
    // L2 eviction policy of the TMA loads of A' and B' and of the TMA stores
    // of C: 0 none, 1 evict first, 2 evict last (see l2_policy).
    uint32_t l2_a, l2_b, l2_c;
    // Work decomposition.  `workers` persistent CTAs (single form) or clusters
    // (pair form).  Worker c first takes the whole-tile (or classic split-K)
    // units c, c+workers, ... < num_units; then, if sk_iters > 0, the
    // stream-K range [c*S/P, (c+1)*S/P) of the S = sk_iters K blocks of tiles
    // sk_tile0 .. tiles-1, cut at tile boundaries into segments.
    int workers;
    int sk_tile0;
    int64_t sk_iters;
    int nseg_max;       // most units that cover one stream-K tile (slots per stream-K tile)
    int sk_slot_base;   // first partial slot of the stream-K segments
    // Tail split: whole tiles from tail_tile0 on are cut along N into
    // tail_split units of BN / tail_split columns, so that a last partial wave
    // of tiles spreads over more workers (no partial sums involved).
    int tail_tile0;
    int tail_split;
    // Several problems in one launch (TileLang tutorial ch. 14, sections 4.3
    // and 4.4).  gmode 0: one GEMM.  1: `groups` batches of the same shape,
    // batch b at element offsets b*a_bs, b*b_bs, b*c_bs (a stride of 0 shares
    // the operand); tiles are numbered batch by batch.  2: grouped: G GEMMs
    // that share K and N, group g owning rows g_row0[g] .. + g_rows[g] of the
    // concatenated A' and C and batch g of B'; its tiles start at g_tile0[g]
    // and span g_tm[g] tile rows.  An operand whose tensor map carries a
    // trailing batch dimension (x_bdim) takes the batch or group index as that
    // coordinate.
    int gmode, groups;
    uint32_t a_bdim, b_bdim, c_bdim;
    int64_t a_bs, b_bs, c_bs;
    int g_tile0[kMaxGroups + 1];
    int g_tm[kMaxGroups];
    int64_t g_row0[kMaxGroups];
    int64_t g_rows[kMaxGroups];
    // Fused output stage (kEpi kernels): out = act(acc + bias), or, gated,
    // out = act(acc_gate + bias) * (acc_up + bias_up).  A gated tile's BN
    // accumulator columns are BN/2 gate columns followed by the same BN/2
    // columns of the up projection: both B' operands land in one stage, so one
    // MMA stream computes both products of the shared A' rows.
    const __half* Bu;         // up projection B' (the strides and batch stride of B')
    const __half* bias;       // fp16 bias, or null
    const __half* bias_up;    // fp16 bias of the up projection, or null
    int64_t bias_bs;          // elements between the bias vectors of consecutive problems / groups
    int act;                  // 0 identity, 1 ReLU, 2 SiLU, 3 GELU (exact, x * Phi(x))
    int gated;
    int bias_rows;            // 1: the bias runs along the kernel view's rows (the swapped form)
};
// (a __grid_constant__ parameter block: at most 4 KB keeps it within every
// launch path's limit)
static_assert(sizeof(KernelParams) <= 4096, "kernel parameters exceed 4 KB");

struct SmemLayout {
    uint32_t a, b, epi, bars;
};

__device__ __forceinline__ SmemLayout smem_layout(const KernelParams& p, uint32_t base)
{
    SmemLayout s;
    s.a = base;
    s.b = s.a + p.stages * kStageABytes;
    s.epi = s.b + p.stages * p.stage_b_bytes;
    s.bars = s.epi + (p.epi_smem ? kEpiBytes : 0u);
    return s;
}

// Barrier block: full[16], empty[16], tmem_full[2], tmem_empty[2], drain,
// fixup, then the TMEM base address, the abort flag and broadcast words.
__device__ __forceinline__ uint32_t bar_full(uint32_t bars, int s) { return bars + 8u * s; }
__device__ __forceinline__ uint32_t bar_empty(uint32_t bars, int s) { return bars + 8u * (kMaxStages + s); }
__device__ __forceinline__ uint32_t bar_tfull(uint32_t bars, int a) { return bars + 8u * (2 * kMaxStages + a); }
__device__ __forceinline__ uint32_t bar_tempty(uint32_t bars, int a) { return bars + 8u * (2 * kMaxStages + 2 + a); }
__device__ __forceinline__ uint32_t bar_drain(uint32_t bars) { return bars + 8u * (2 * kMaxStages + 4); }
__device__ __forceinline__ uint32_t bar_fix(uint32_t bars) { return bars + 8u * (2 * kMaxStages + 5); }
// Failure-detection test only: a barrier nothing ever arrives on (see test_stall).
__device__ __forceinline__ uint32_t bar_never(uint32_t bars) { return bars + 8u * (2 * kMaxStages + 6); }
constexpr uint32_t kTmemSlotOff = 8u * (2 * kMaxStages + 7);
constexpr uint32_t kAbortOff = kTmemSlotOff + 4;
constexpr uint32_t kFlagOff = kTmemSlotOff + 8;
constexpr uint32_t kOkOff = kTmemSlotOff + 12;   // two words, indexed by accumulator
constexpr uint64_t kDrainTimeoutNs = 10000000ull;

// One unit of a worker's list: K blocks [kb0, kb1) of one output tile.  A unit
// that covers the whole K range is stored directly (slot < 0).  Otherwise it
// leaves an fp32 partial in workspace slot `slot`; `expected` units cover the
// tile, and the last of them to finish adds all partials in K order.
struct Unit {
    int tile, m_blk, n_blk, kb0, kb1, slot, expected;
    int g;       // batch or group of the tile
    int seg;     // index of this unit among the units covering its tile, in K order
    int slot0;   // slot of the tile's first unit: the idx-th (K order) one is slot0 + idx
    int bn;      // columns of this unit (BN, or BN / tail_split for a tail piece)
    int n_off;   // first column of this unit inside its tile
};

// Tile -> (row block, column block).  Tiles are numbered in panels of `panel`
// tile-rows; inside a panel the row index moves fastest, so CTAs running at the
// same time share B columns and a few A row-blocks in L2 (the grouped program
// ordering of the Triton page; the C500 review's panel rasterisation, section
// 10).  The ordering is only a locality hint.
template <bool kMulti>
__device__ __forceinline__ void tile_coords(const KernelParams& p, int tile, int& g, int& m_blk, int& n_blk)
{
    int t = tile, tm = p.tiles_m;
    g = 0;
    if (!kMulti) {
    } else if (p.gmode == 1) {   // batches of tiles_m x tiles_n tiles
        const int per = p.tiles_m * p.tiles_n;
        g = tile / per;
        t = tile - g * per;
    } else if (p.gmode == 2) {   // groups of g_tm[g] x tiles_n tiles
        while (g + 1 < p.groups && tile >= p.g_tile0[g + 1]) ++g;
        t = tile - p.g_tile0[g];
        tm = p.g_tm[g];
    }
    const int per_panel = p.panel * p.tiles_n;
    const int panel = t / per_panel;
    const int r = t - panel * per_panel;
    const int rows = min(p.panel, tm - panel * p.panel);
    m_blk = panel * p.panel + r % rows;
    n_blk = r / rows;
}

// Stream-K (TileLang tutorial ch. 14, section 4.2: split the total K
// iterations evenly over the processors, fix up only the tiles that got cut).
// Worker c's range starts at K block c*S/P of the stream-K tiles.
__device__ __forceinline__ int64_t sk_start(const KernelParams& p, int c)
{
    return static_cast<int64_t>(c) * p.sk_iters / p.workers;
}

// The worker whose range holds stream-K block x: the largest c with
// sk_start(c) <= x, i.e. ceil((x+1)*P/S) - 1.
__device__ __forceinline__ int sk_worker(const KernelParams& p, int64_t x)
{
    const int64_t c = ((x + 1) * p.workers + p.sk_iters - 1) / p.sk_iters - 1;
    return static_cast<int>(c < p.workers - 1 ? c : p.workers - 1);
}

__device__ __forceinline__ int classic_units(const KernelParams& p, int cid)
{
    return cid < p.num_units ? (p.num_units - cid + p.workers - 1) / p.workers : 0;
}

__device__ __forceinline__ int units_of_worker(const KernelParams& p, int cid)
{
    int n = classic_units(p, cid);
    if (p.sk_iters > 0) {
        const int64_t s0 = sk_start(p, cid), s1 = sk_start(p, cid + 1);
        if (s1 > s0) n += static_cast<int>((s1 - 1) / p.kblocks - s0 / p.kblocks + 1);
    }
    return n;
}

// The i-th unit of worker `cid`: whole tiles or classic split-K units first
// (u = cid, cid + P, ...; the units of one split tile are consecutive), then
// the worker's stream-K segments in K order.
template <bool kMulti>
__device__ __forceinline__ Unit unit_at(const KernelParams& p, int cid, int i)
{
    Unit w;
    w.slot = -1;
    w.slot0 = -1;
    w.expected = 1;
    w.seg = 0;
    w.bn = p.BN;
    w.n_off = 0;
    const int nc = classic_units(p, cid);
    if (i < nc) {
        const int u = cid + i * p.workers;
        if (u >= p.tail_tile0) {
            const int v = u - p.tail_tile0;
            w.tile = p.tail_tile0 + v / p.tail_split;
            w.bn = p.BN / p.tail_split;
            w.n_off = (v % p.tail_split) * w.bn;
            w.kb0 = 0;
            w.kb1 = p.kblocks;
        } else {
            // Classic split-K units are numbered K segment first (unit u: tile
            // u mod tiles, segment u / tiles), so the units in flight at once
            // cover the same K range of neighbouring tiles and read the same
            // operand rows together (16 x 16384 x 8192, 2 segments: 53.2
            // against 56.3 us per call with the tile-major order).
            const int ntl = p.num_units / p.splits;   // (classic split-K: units = tiles * splits)
            w.tile = u % ntl;
            const int split = u / ntl;
            w.kb0 = static_cast<int>(static_cast<int64_t>(split) * p.kblocks / p.splits);
            w.kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * p.kblocks / p.splits);
            if (p.splits > 1) {
                w.slot0 = w.tile * p.splits;
                w.slot = w.slot0 + split;
                w.expected = p.splits;
                w.seg = split;
            }
        }
    } else {
        const int j = i - nc;
        const int64_t s0 = sk_start(p, cid), s1 = sk_start(p, cid + 1);
        const int64_t t0 = s0 / p.kblocks + j;
        w.kb0 = (j == 0) ? static_cast<int>(s0 % p.kblocks) : 0;
        w.kb1 = (t0 == (s1 - 1) / p.kblocks) ? static_cast<int>((s1 - 1) % p.kblocks) + 1 : p.kblocks;
        w.tile = p.sk_tile0 + static_cast<int>(t0);
        if (w.kb0 != 0 || w.kb1 != p.kblocks) {
            const int first = sk_worker(p, t0 * p.kblocks);
            w.expected = sk_worker(p, t0 * p.kblocks + p.kblocks - 1) - first + 1;
            w.seg = cid - first;
            w.slot0 = p.sk_slot_base + static_cast<int>(t0) * p.nseg_max;
            w.slot = w.slot0 + w.seg;
        }
    }
    tile_coords<kMulti>(p, w.tile, w.g, w.m_blk, w.n_blk);
    return w;
}

// Where one unit's problem lives: the A'/C row of its row 0 (groups are
// concatenated along rows), the first row past its problem, the trailing
// (batch) coordinates of the three tensor maps, and the bases the gather and
// masked paths index from.
struct UnitGeom {
    int64_t a_row, row_lim;
    int32_t az, bz, cz;
    const __half* A;
    const __half* B;
    const __half* Bu;   // gated fused stage only
    __half* C;
};

template <bool kMulti>
__device__ __forceinline__ UnitGeom unit_geom(const KernelParams& p, const Unit& w)
{
    UnitGeom u;
    const int64_t g = w.g;
    u.a_row = 0;
    u.row_lim = p.M;
    u.az = u.bz = u.cz = 0;
    u.A = p.A;
    u.B = p.B;
    u.Bu = p.Bu;
    u.C = p.C;
    if (!kMulti) {
    } else if (p.gmode == 1) {
        u.az = u.bz = u.cz = w.g;
        u.A = p.A + g * p.a_bs;
        u.B = p.B + g * p.b_bs;
        u.Bu = p.Bu + g * p.b_bs;
        u.C = p.C + g * p.c_bs;
    } else if (p.gmode == 2) {
        u.a_row = p.g_row0[w.g];
        u.row_lim = p.g_row0[w.g] + p.g_rows[w.g];
        u.bz = w.g;
        u.B = p.B + g * p.b_bs;
        u.Bu = p.Bu + g * p.b_bs;
    }
    return u;
}

// TMA loads of one slot, single or pair form, with the map's trailing batch
// coordinate z when it has one; `hk` is the L2 eviction policy kind of the
// operand (0: none; see l2_policy).
template <bool kPair>
__device__ __forceinline__ void tma2(uint32_t d, const void* m, int32_t x, int32_t y, uint32_t bar, uint32_t hk)
{
    if (hk) {
        if (kPair)
            tma_load_2d_pair_hint(d, m, x, y, bar, l2_policy(hk));
        else
            tma_load_2d_hint(d, m, x, y, bar, l2_policy(hk));
    } else if (kPair) {
        tma_load_2d_pair(d, m, x, y, bar);
    } else {
        tma_load_2d(d, m, x, y, bar);
    }
}
template <bool kPair>
__device__ __forceinline__ void tma3(uint32_t d, const void* m, int32_t x, int32_t y, int32_t z, uint32_t bar,
                                     uint32_t hk)
{
    if (hk) {
        if (kPair)
            tma_load_3d_pair_hint(d, m, x, y, z, bar, l2_policy(hk));
        else
            tma_load_3d_hint(d, m, x, y, z, bar, l2_policy(hk));
    } else if (kPair) {
        tma_load_3d_pair(d, m, x, y, z, bar);
    } else {
        tma_load_3d(d, m, x, y, z, bar);
    }
}
template <bool kPair>
__device__ __forceinline__ void tma5(uint32_t d, const void* m, int32_t x, int32_t y, int32_t z, int32_t v, int32_t u,
                                     uint32_t bar, uint32_t hk)
{
    if (hk) {
        if (kPair)
            tma_load_5d_pair_hint(d, m, x, y, z, v, u, bar, l2_policy(hk));
        else
            tma_load_5d_hint(d, m, x, y, z, v, u, bar, l2_policy(hk));
    } else if (kPair) {
        tma_load_5d_pair(d, m, x, y, z, v, u, bar);
    } else {
        tma_load_5d(d, m, x, y, z, v, u, bar);
    }
}
template <bool kPair>
__device__ __forceinline__ void tma4(uint32_t d, const void* m, int32_t x, int32_t y, int32_t z, int32_t v,
                                     uint32_t bar, uint32_t hk)
{
    if (hk) {
        if (kPair)
            tma_load_4d_pair_hint(d, m, x, y, z, v, bar, l2_policy(hk));
        else
            tma_load_4d_hint(d, m, x, y, z, v, bar, l2_policy(hk));
    } else if (kPair) {
        tma_load_4d_pair(d, m, x, y, z, v, bar);
    } else {
        tma_load_4d(d, m, x, y, z, v, bar);
    }
}

// A' rows row .. row+127 of one 64-wide K slot: K-major one box (k, row);
// MN-major one 3-D box (0, k, row/64) or two 2-D boxes (row, k) and (row+64, k).
template <bool kPair>
__device__ __forceinline__ void load_a_slot(const KernelParams& p, uint32_t sa, int32_t k0, int64_t row, int32_t z,
                                            bool a_mn, bool a_3d, bool bd, uint32_t bar)
{
    const int32_t r = static_cast<int32_t>(row);
    if (!a_mn) {
        if (bd)
            tma3<kPair>(sa, &p.tmA, k0, r, z, bar, p.l2_a);
        else
            tma2<kPair>(sa, &p.tmA, k0, r, bar, p.l2_a);
    } else if (a_3d) {
        if (bd)
            tma4<kPair>(sa, &p.tmA, 0, k0, r >> 6, z, bar, p.l2_a);
        else
            tma3<kPair>(sa, &p.tmA, 0, k0, r >> 6, bar, p.l2_a);
    } else {
        for (int j = 0; j < 2; ++j) {
            if (bd)
                tma3<kPair>(sa + j * 8192, &p.tmA, r + 64 * j, k0, z, bar, p.l2_a);
            else
                tma2<kPair>(sa + j * 8192, &p.tmA, r + 64 * j, k0, bar, p.l2_a);
        }
    }
}

// B' columns col .. col+bcols-1 of one slot through map `tmb`: K-major one box
// (k, col) of the map's width; MN-major one 3-D box (0, k, col/64) or one 2-D
// box (col, k) per 64 columns.
template <bool kPair>
__device__ __forceinline__ void load_b_slot(const KernelParams& p, const CUtensorMap* tmb, uint32_t sb, int32_t k0,
                                            int64_t col, int32_t z, int bcols, bool b_mn, bool b_3d, bool bd,
                                            uint32_t bar)
{
    const int32_t c = static_cast<int32_t>(col);
    if (!b_mn) {
        if (bd)
            tma3<kPair>(sb, tmb, k0, c, z, bar, p.l2_b);
        else
            tma2<kPair>(sb, tmb, k0, c, bar, p.l2_b);
    } else if (b_3d) {
        if (bd)
            tma4<kPair>(sb, tmb, 0, k0, c >> 6, z, bar, p.l2_b);
        else
            tma3<kPair>(sb, tmb, 0, k0, c >> 6, bar, p.l2_b);
    } else {
        for (int j = 0; j < bcols / 64; ++j) {
            if (bd)
                tma3<kPair>(sb + j * 8192, tmb, c + 64 * j, k0, z, bar, p.l2_b);
            else
                tma2<kPair>(sb + j * 8192, tmb, c + 64 * j, k0, bar, p.l2_b);
        }
    }
}

// Both K blocks kb, kb+1 of a barrier phase in one copy per operand, into the
// phase's two consecutive slots (sa, sb: the first slot's A' and B' bases);
// the A' copy when do_a, the B' copy when do_b.
// A' rows row .. row+127; B' columns col .. col + (the box width of tmb).
template <bool kPair>
__device__ __forceinline__ void load_two_k_blocks(const KernelParams& p, const CUtensorMap* tmb, uint32_t sa,
                                                  uint32_t sb, int32_t kb, int64_t row, int64_t col, int32_t az,
                                                  int32_t bz, bool a_mn, bool b_mn, bool a_bd, bool b_bd, uint32_t bar,
                                                  bool do_a, bool do_b)
{
    const int32_t r = static_cast<int32_t>(row), c = static_cast<int32_t>(col);
    if (do_a) {
        if (!a_mn) {
            if (a_bd)
                tma4<kPair>(sa, &p.tmA2k, 0, r, kb, az, bar, p.l2_a);
            else
                tma3<kPair>(sa, &p.tmA2k, 0, r, kb, bar, p.l2_a);
        } else if (a_bd) {
            tma5<kPair>(sa, &p.tmA2k, 0, 0, r >> 6, kb, az, bar, p.l2_a);
        } else {
            tma4<kPair>(sa, &p.tmA2k, 0, 0, r >> 6, kb, bar, p.l2_a);
        }
    }
    if (do_b) {
        if (!b_mn) {
            if (b_bd)
                tma4<kPair>(sb, tmb, 0, c, kb, bz, bar, p.l2_b);
            else
                tma3<kPair>(sb, tmb, 0, c, kb, bar, p.l2_b);
        } else if (b_bd) {
            tma5<kPair>(sb, tmb, 0, 0, c >> 6, kb, bz, bar, p.l2_b);
        } else {
            tma4<kPair>(sb, tmb, 0, 0, c >> 6, kb, bar, p.l2_b);
        }
    }
}

__device__ __forceinline__ void raise_abort(const KernelParams& p, volatile int* abort)
{
    *abort = 1;
    if (p.status) atomicExch(p.status, kStatusTimeout);
}

template <bool kPair>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const volatile int* abort, uint64_t tmo)
{
    return kPair ? mbar_wait_cluster(bar, parity, abort, tmo) : mbar_wait(bar, parity, abort, tmo);
}

// Bytes [sh, sh+16) of the 32-byte little-endian value w1:w0 (sh even, 2..14).
__device__ __forceinline__ uint4 funnel16(const uint4& w0, const uint4& w1, uint32_t sh)
{
    const uint32_t s = (sh & 3u) * 8u;
    uint32_t x0, x1, x2, x3, x4;
    switch (sh >> 2) {
    case 0: x0 = w0.x, x1 = w0.y, x2 = w0.z, x3 = w0.w, x4 = w1.x; break;
    case 1: x0 = w0.y, x1 = w0.z, x2 = w0.w, x3 = w1.x, x4 = w1.y; break;
    case 2: x0 = w0.z, x1 = w0.w, x2 = w1.x, x3 = w1.y, x4 = w1.z; break;
    default: x0 = w0.w, x1 = w1.x, x2 = w1.y, x3 = w1.z, x4 = w1.w; break;
    }
    return make_uint4(__funnelshift_r(x0, x1, s), __funnelshift_r(x1, x2, s), __funnelshift_r(x2, x3, s),
                      __funnelshift_r(x3, x4, s));
}

// Keep the first `nvalid` (< 8) fp16 values of a 16-byte chunk, zero the rest.
__device__ __forceinline__ uint4 keep_first(uint4 r, int nvalid)
{
    const uint32_t nb = 2u * static_cast<uint32_t>(nvalid);
    auto k = [nb](uint32_t w, uint32_t i) -> uint32_t {
        return (4u * i + 4u <= nb) ? w : ((4u * i >= nb) ? 0u : (w & 0xFFFFu));
    };
    return make_uint4(k(r.x, 0), k(r.y, 1), k(r.z, 2), k(r.w, 3));
}

// Debug bounds check of one access of `bytes` at address a against span
// `which`.  A gathered 16-byte word is read whole to reach the elements inside
// it, so for a word (`word`) it is enough that it overlaps the span; every
// other access must lie inside.  Off (the default) it is one uniform test.
__device__ __forceinline__ bool bounds_ok(const KernelParams& p, int which, uintptr_t a, uint32_t bytes, bool word)
{
    if (!p.debug_bounds) return true;
    const uintptr_t lo = p.span_lo[which], hi = p.span_hi[which];
    const bool ok = word ? (a < hi && a + bytes > lo) : (a >= lo && a + bytes <= hi);
    if (!ok && p.status) atomicExch(p.status, kStatusBounds);
    return ok;
}

// Eight elements along a non-unit `step` from element offset `off`; the first
// `nvalid` are loaded one by one, the rest are zero.
__device__ __forceinline__ uint4 load8_strided(const KernelParams& p, int which, const __half* base, int64_t off,
                                               int64_t step, int nvalid)
{
    const uint16_t* q = reinterpret_cast<const uint16_t*>(base) + off;
    uint32_t v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        v[e] = (e < nvalid && bounds_ok(p, which, reinterpret_cast<uintptr_t>(q + e * step), 2, false))
                   ? static_cast<uint32_t>(ld_nc_u16(q + e * step))
                   : 0u;
    return make_uint4(v[0] | (v[1] << 16), v[2] | (v[3] << 16), v[4] | (v[5] << 16), v[6] | (v[7] << 16));
}

__device__ __forceinline__ int clamp8(int64_t remaining)
{
    return remaining >= 8 ? 8 : (remaining <= 0 ? 0 : static_cast<int>(remaining));
}

// Chunks each producer thread keeps in flight while gathering with a non-unit
// stride (unit-stride operands go row by row, below).
constexpr int kGatherBatch = 4;

// Gather one operand tile (rows = MN extent `rows_tile`, 64 K columns) into the
// 128B-swizzled layout the UMMA descriptor expects.  K-major: row r (128 B) at
// r*128, its 16-byte chunk j at ((j ^ (r & 7)) << 4).  MN-major: atom column a
// (64 MN elements) at a*8192, K row r at r*128, chunk j swizzled the same way.
//
// A chunk is 8 consecutive elements of the operand's contiguous dimension; the
// first `nvalid` lie inside the view (row < extent, k < K), the rest are
// zero-filled.  With a unit stride the chunk is assembled from the aligned
// 16-byte word holding its first element plus, only when a valid element lies
// in it, the next word; bytes of those words outside the view are discarded.
// A 16-byte-aligned word that holds a valid element cannot cross that
// element's page, so no load can fault.  Chunks are handled four at a time:
// first every load is issued, then the words are shifted into place and
// stored, so a thread keeps up to 8 loads in flight (more spills registers).
// Unit-stride operands, row by row: each thread fills whole 128-byte rows of
// the swizzled tile (64 consecutive elements of the contiguous dimension: a
// K-major row, or one K row of an MN-major atom column).  The row's elements
// start at any 2-byte-aligned address; the thread loads the aligned 16-byte
// words that hold valid elements (at most 9, the same rule as above, so no
// load can fault), then funnel-shifts them into the row's 8 chunks.  One
// address computation per row instead of per chunk, and two rows in flight.
__device__ __forceinline__ int clamp64(int64_t remaining)
{
    return remaining >= 64 ? 64 : (remaining <= 0 ? 0 : static_cast<int>(remaining));
}

// Shift a row's 36 loaded words left by `sh` bytes (even, 0..14) and store its
// 8 chunks: word o of the row is bytes [4o + sh, 4o + sh + 4) of the words,
// i.e. a funnel shift of words o + sh/4 and o + sh/4 + 1 by 8*(sh%4) bits.
// The word offset sh/4 is applied as two levels of selects (by 1 word, then
// by 2), so lanes whose rows have different offsets take the same
// instructions (no divergent branch per chunk).
__device__ __forceinline__ void shift_store_row(const uint4* wv, uint32_t sh, int nv, uint32_t rowaddr, int rk)
{
    uint32_t w[36];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        w[4 * i] = wv[i].x;
        w[4 * i + 1] = wv[i].y;
        w[4 * i + 2] = wv[i].z;
        w[4 * i + 3] = wv[i].w;
    }
    const bool d1 = (sh & 4u) != 0, d2 = (sh & 8u) != 0;
    const uint32_t s = (sh & 3u) * 8u;
#pragma unroll
    for (int k = 0; k < 35; ++k) w[k] = d1 ? w[k + 1] : w[k];
#pragma unroll
    for (int k = 0; k < 33; ++k) w[k] = d2 ? w[k + 2] : w[k];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint4 c = make_uint4(__funnelshift_r(w[4 * j], w[4 * j + 1], s), __funnelshift_r(w[4 * j + 1], w[4 * j + 2], s),
                             __funnelshift_r(w[4 * j + 2], w[4 * j + 3], s),
                             __funnelshift_r(w[4 * j + 3], w[4 * j + 4], s));
        const int cv = clamp8(nv - 8 * j);
        if (cv < 8) c = keep_first(c, cv);   // (cv <= 0 zeroes the chunk)
        st_smem_v4(rowaddr + ((j ^ (rk & 7)) << 4), c);
    }
}

// Rows each producer thread has in flight (9 loads each) in the unit-stride gather.
constexpr int kGatherRows = 2;

__device__ __forceinline__ void gather_rows_unit(const KernelParams& p, int which, const __half* base,
                                                 int64_t s_mn, int64_t s_k, int64_t MN,
                                                 int64_t K, int64_t mn0, int64_t k0, int rows_tile, bool mn_major,
                                                 uint32_t dst, int t)
{
    const int nrows = rows_tile;   // K-major: MN rows; MN-major: (rows_tile / 64) atoms x 64 K rows
    const uintptr_t b = reinterpret_cast<uintptr_t>(base);
    for (int r0 = t; r0 < nrows; r0 += kGatherRows * kProducerThreads) {
        uint4 wv[kGatherRows][9];
        uint32_t sh[kGatherRows], rowaddr[kGatherRows];
        int nv[kGatherRows], rk[kGatherRows];
#pragma unroll
        for (int q = 0; q < kGatherRows; ++q) {
            const int rr = r0 + q * kProducerThreads;
            nv[q] = 0;
            sh[q] = 0;
            rk[q] = 0;
            rowaddr[q] = 0;
            if (rr < nrows) {
                int64_t off;
                if (!mn_major) {
                    const int64_t mn = mn0 + rr;
                    nv[q] = (mn < MN) ? clamp64(K - k0) : 0;
                    off = mn * s_mn + k0;   // s_k == 1
                    rk[q] = rr;
                    rowaddr[q] = dst + rr * 128;
                } else {
                    const int a = rr >> 6, r = rr & 63;   // atom column a, K row r
                    const int64_t k = k0 + r, mn = mn0 + 64 * a;
                    nv[q] = (k < K) ? clamp64(MN - mn) : 0;
                    off = k * s_k + mn;   // s_mn == 1
                    rk[q] = r;
                    rowaddr[q] = dst + a * 8192 + r * 128;
                }
                const uintptr_t addr = b + 2 * static_cast<uintptr_t>(off);
                sh[q] = static_cast<uint32_t>(addr & 15u);
                const uintptr_t a0 = addr - sh[q];
                // words holding valid elements (none when the row is outside the view)
                const int nw = nv[q] > 0 ? static_cast<int>((sh[q] + 2u * static_cast<uint32_t>(nv[q]) + 15u) / 16u) : 0;
#pragma unroll
                for (int i = 0; i < 9; ++i)
                    wv[q][i] = (i < nw && bounds_ok(p, which, a0 + 16u * i, 16, true))
                                   ? ld_nc_v4(reinterpret_cast<const void*>(a0 + 16u * i))
                                   : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int q = 0; q < kGatherRows; ++q) {
            if (r0 + q * kProducerThreads >= nrows) break;
            shift_store_row(wv[q], sh[q], nv[q], rowaddr[q], rk[q]);
        }
    }
}

__device__ __forceinline__ void gather_tile(const KernelParams& p, int which, const __half* base, int64_t s_mn,
                                            int64_t s_k,
                                            int64_t MN, int64_t K, int64_t mn0, int64_t k0,
                                            int rows_tile, bool mn_major, uint32_t dst, int t)
{
    if ((mn_major ? s_mn : s_k) == 1) {
        gather_rows_unit(p, which, base, s_mn, s_k, MN, K, mn0, k0, rows_tile, mn_major, dst, t);
        return;
    }
    const int chunks = rows_tile * 8;   // 16-byte chunks in the tile
    const int iters = (chunks + kProducerThreads - 1) / kProducerThreads;
    const int atoms = rows_tile / 64;
    const int64_t step = mn_major ? s_mn : s_k;
    const uintptr_t b = reinterpret_cast<uintptr_t>(base);
    for (int i0 = 0; i0 < iters; i0 += kGatherBatch) {
        uint4 w0[kGatherBatch], w1[kGatherBatch];
        uint32_t addr[kGatherBatch], sh[kGatherBatch];
        int nv[kGatherBatch];
#pragma unroll
        for (int i = 0; i < kGatherBatch; ++i) {
            nv[i] = 0;
            const int c = t + kProducerThreads * (i0 + i);
            if (i0 + i < iters && c < chunks) {
                const int j = c & 7;
                int64_t mn, k;
                if (!mn_major) {
                    const int r = c >> 3;
                    mn = mn0 + r;
                    k = k0 + 8 * j;
                    nv[i] = (mn < MN) ? clamp8(K - k) : 0;
                    addr[i] = dst + r * 128 + ((j ^ (r & 7)) << 4);
                } else {
                    const int a = (c >> 3) % atoms;
                    const int r = (c >> 3) / atoms;
                    mn = mn0 + 64 * a + 8 * j;
                    k = k0 + r;
                    nv[i] = (k < K) ? clamp8(MN - mn) : 0;
                    addr[i] = dst + a * 8192 + r * 128 + ((j ^ (r & 7)) << 4);
                }
                sh[i] = 0;
                w0[i] = make_uint4(0u, 0u, 0u, 0u);
                w1[i] = w0[i];
                if (nv[i] > 0) {
                    const int64_t off = mn * s_mn + k * s_k;
                    if (step == 1) {
                        const uintptr_t a = b + 2 * static_cast<uintptr_t>(off);
                        sh[i] = static_cast<uint32_t>(a & 15u);
                        const uintptr_t a0 = a - sh[i];
                        const bool two = sh[i] != 0 && sh[i] + 2u * static_cast<uint32_t>(nv[i]) > 16u;
                        if (bounds_ok(p, which, a0, 16, true)) w0[i] = ld_nc_v4(reinterpret_cast<const void*>(a0));
                        if (two && bounds_ok(p, which, a0 + 16, 16, true))
                            w1[i] = ld_nc_v4(reinterpret_cast<const void*>(a0 + 16));
                    } else {
                        w0[i] = load8_strided(p, which, base, off, step, nv[i]);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kGatherBatch; ++i) {
            if (i0 + i < iters && t + kProducerThreads * (i0 + i) < chunks) {
                uint4 r = (sh[i] != 0) ? funnel16(w0[i], w1[i], sh[i]) : w0[i];
                if (nv[i] < 8) r = keep_first(r, nv[i]);
                st_smem_v4(addr[i], r);
            }
        }
    }
}

// Write a warp's staged 32 x 64 box (swizzled like a TMA box; `ncols` of its
// columns hold output) to C rows crow .. crow+31, columns n .. n+ncols-1, row by
// row: lane l writes columns 2l and 2l+1, as one 4-byte store where the address
// allows, so each store instruction covers 128 contiguous bytes of a row.
// Rows at or past row_lim and columns at or past N are not written.
__device__ __forceinline__ void store_box_rows(const KernelParams& p, __half* C, int64_t row_lim, uint32_t buf,
                                               int64_t crow, int64_t n, int ncols)
{
    const int lane = threadIdx.x & 31;
    const int c = 2 * lane;
    const int64_t nn = n + c;
    const bool in0 = c < ncols && nn < p.N, in1 = c + 1 < ncols && nn + 1 < p.N;
    const int j = c >> 3;   // 16-byte chunk of the box row
    uint16_t* base = reinterpret_cast<uint16_t*>(C) + nn;
    for (int r = 0; r < 32; ++r) {
        const int64_t m = crow + r;
        if (m >= row_lim) break;
        const uint32_t v = ld_smem_u32(buf + r * 128 + ((j ^ (r & 7)) << 4) + (c & 7) * 2);
        uint16_t* q = base + m * p.c_sm;
        const uintptr_t qa = reinterpret_cast<uintptr_t>(q);
        if (in1 && (qa & 3u) == 0) {
            if (bounds_ok(p, kSpanC, qa, 4, false)) *reinterpret_cast<uint32_t*>(q) = v;
        } else {
            if (in0 && bounds_ok(p, kSpanC, qa, 2, false)) q[0] = static_cast<uint16_t>(v);
            if (in1 && bounds_ok(p, kSpanC, qa + 2, 2, false)) q[1] = static_cast<uint16_t>(v >> 16);
        }
    }
}

__device__ __forceinline__ uint16_t half_bits(const uint32_t* h, int c)
{
    return static_cast<uint16_t>(h[c >> 1] >> ((c & 1) * 16));
}

// Store 16 fp16 values (h[8]) of output row m, columns n..n+15, with bounds
// checks on m and on every column.
__device__ __forceinline__ void store_piece_masked(const KernelParams& p, __half* C, int64_t m_lim, int64_t m, int64_t n,
                                                   const uint32_t* h)
{
    if (m >= m_lim || n >= p.N) return;
    uint16_t* row = reinterpret_cast<uint16_t*>(C) + m * p.c_sm;
    if (p.c_sn == 1) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t nn = n + 8 * j;
            uint16_t* q = row + nn;
            if (nn + 8 <= p.N && (reinterpret_cast<uintptr_t>(q) & 15u) == 0) {
                if (bounds_ok(p, kSpanC, reinterpret_cast<uintptr_t>(q), 16, false))
                    *reinterpret_cast<uint4*>(q) = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (nn + e < p.N && bounds_ok(p, kSpanC, reinterpret_cast<uintptr_t>(q + e), 2, false))
                        q[e] = half_bits(h, 8 * j + e);
            }
        }
    } else {
        uint16_t* q = row + n * p.c_sn;
        const int64_t lim = p.N - n;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            if (c < lim && bounds_ok(p, kSpanC, reinterpret_cast<uintptr_t>(q), 2, false)) *q = half_bits(h, c);
            q += p.c_sn;
        }
    }
}

__device__ __forceinline__ void convert16(const uint32_t* r, uint32_t* h)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = pack_half2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
}

// sacc[i] += the fp32 accumulator column taddr + i of this thread's lane.
__device__ __forceinline__ void add_tmem16(uint32_t taddr, float* sacc)
{
    uint32_t v[16];
    tmem_ld_x16(taddr, v);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) sacc[i] += __uint_as_float(v[i]);
}

// ---------------------------------------------------------------------------
// Fused output stage.  The pages name bias and activation fusion into the
// GEMM's output stage (TileLang tutorial ch. 14, section 6.3, item 4; AI-infra
// page, section 05) and a gate/up GEMM that fuses two projections with the
// activation and the multiply (C500 review, section 17.3).  Everything runs in
// fp32 on the accumulator values, with one rounding to fp16 at the store.

// act(x): 1 ReLU (x < 0 -> 0, NaN kept), 2 SiLU x / (1 + e^-x),
// 3 GELU x * Phi(x) with Phi(x) = erfc(-x / sqrt 2) / 2; otherwise identity.
__device__ __forceinline__ float act_apply(int act, float x)
{
    switch (act) {
    case 1: return x < 0.f ? 0.f : x;
    case 2: return x / (1.f + expf(-x));
    case 3: return x * (0.5f * erfcf(-x * 0.70710678118654752f));
    default: return x;
    }
}

__device__ __forceinline__ float half_lo(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w))); }
__device__ __forceinline__ float half_hi(uint32_t w)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// v[i] = b[n + i] for the 16 columns n .. n+15 (0 past N, or without a bias).
__device__ __forceinline__ void load_bias16(const __half* b, int64_t n, int64_t N, float* v)
{
    if (b == nullptr) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
        return;
    }
    const __half* q = b + n;
    if (n + 16 <= N && (reinterpret_cast<uintptr_t>(q) & 15u) == 0) {
        const uint4 x0 = __ldg(reinterpret_cast<const uint4*>(q));
        const uint4 x1 = __ldg(reinterpret_cast<const uint4*>(q) + 1);
        const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = half_lo(w[i]);
            v[2 * i + 1] = half_hi(w[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = (n + i < N) ? __half2float(q[i]) : 0.f;
    }
}

// v = act(v + bias) for 16 sums of kernel columns n .. n+15 of one row: the
// bias along the columns, or (bias_rows) the row's own value `brow`.
__device__ __forceinline__ void epi_finish16(const KernelParams& p, const __half* bias, float brow, int64_t n, float* v)
{
    float b[16];
    if (p.bias_rows) {
#pragma unroll
        for (int i = 0; i < 16; ++i) b[i] = brow;
    } else {
        load_bias16(bias, n, p.N, b);
    }
    const int act = p.act;
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = act_apply(act, v[i] + b[i]);
}

// Gated: g = act(g + bias) * (u + bias_up) for columns n .. n+15.
__device__ __forceinline__ void epi_gated16(const KernelParams& p, const __half* bias, const __half* bias_up, int64_t n,
                                            float* g, const float* u)
{
    float bg[16], bu[16];
    load_bias16(bias, n, p.N, bg);
    load_bias16(bias_up, n, p.N, bu);
    const int act = p.act;
#pragma unroll
    for (int i = 0; i < 16; ++i) g[i] = act_apply(act, g[i] + bg[i]) * (u[i] + bu[i]);
}

// One 16-column piece of a warp's 32 output rows (h: this lane's 8 packed
// pairs): into the warp's swizzled staging buffer, written out by a TMA store
// every four pieces (64 columns) and after the last one, or by masked stores.
template <bool kMulti>
__device__ __forceinline__ void emit_piece(const KernelParams& p, const SmemLayout& L, const UnitGeom& ug, int piece,
                                           int npieces, const uint32_t* h, int64_t m0, int64_t n0, int64_t crow,
                                           bool ctma, uint32_t& buf, uint32_t& group_count)
{
    const int lane = threadIdx.x & 31;
    const int q = (threadIdx.x >> 5) & 3;
    if (ctma || p.c_stage) {
        const int j0 = (piece & 3) * 2;   // 16-byte chunk inside the 128-byte row
        if ((piece & 3) == 0) {
            buf = L.epi + (q * 2 + (group_count & 1u)) * kEpiBufBytes;
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
        }
        st_smem_v4(buf + lane * 128 + ((j0 ^ (lane & 7)) << 4), make_uint4(h[0], h[1], h[2], h[3]));
        st_smem_v4(buf + lane * 128 + (((j0 + 1) ^ (lane & 7)) << 4), make_uint4(h[4], h[5], h[6], h[7]));
        if (!ctma && ((piece & 3) == 3 || piece == npieces - 1)) {
            __syncwarp();
            store_box_rows(p, ug.C, ug.row_lim, buf, crow, n0 + 16 * (piece & ~3), 16 * ((piece & 3) + 1));
            __syncwarp();   // the box is read before the next piece overwrites it
        } else if ((piece & 3) == 3 || piece == npieces - 1) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (crow < ug.row_lim) {
                    const int32_t xn = static_cast<int32_t>(n0 + 16 * (piece & ~3));
                    if (kMulti && p.c_bdim)
                        tma_store_3d_l2(&p.tmC, buf, xn, static_cast<int32_t>(crow), ug.cz, p.l2_c);
                    else
                        tma_store_2d_l2(&p.tmC, buf, xn, static_cast<int32_t>(crow), p.l2_c);
                }
                bulk_commit_group();
            }
            ++group_count;
        }
    } else {
        store_piece_masked(p, ug.C, ug.row_lim, ug.a_row + m0 + 32 * q + lane, n0 + 16 * piece, h);
    }
}

// Whole-tile epilogue with the fused output stage: `ow` output columns from
// n0 (gated: the accumulator's first ow columns are the gate sums, the next
// ow the up sums of the same output columns).
template <bool kPair, bool kMulti>
__device__ __forceinline__ void fused_tile_epilogue(const KernelParams& p, const SmemLayout& L, const UnitGeom& ug,
                                                   const __half* bias, const __half* bias_up, float brow,
                                                   uint32_t taddr, uint32_t tempty, int64_t m0, int64_t n0, int ow,
                                                   bool gated, int64_t crow, bool ctma, uint32_t& group_count)
{
    const int lane = threadIdx.x & 31;
    const int npieces = ow / 16;
    uint32_t buf = 0;
    auto release = [&]() {   // the accumulator is in registers: the MMA may reuse it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            if (kPair)
                mbar_arrive_cluster(tempty);
            else
                mbar_arrive(tempty);
        }
    };
    // One output piece per TMEM wait: the activation's inlined math needs the
    // registers that more accumulator columns in flight would hold.
    for (int piece = 0; piece < npieces; ++piece) {
        const int64_t n = n0 + 16 * piece;
        uint32_t r[32];
        tmem_ld_x16(taddr + 16 * piece, r);
        if (gated) tmem_ld_x16(taddr + ow + 16 * piece, r + 16);
        tmem_wait_ld();
        if (piece == npieces - 1) release();
        float g[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) g[i] = __uint_as_float(r[i]);
        if (gated) {
            float u[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) u[i] = __uint_as_float(r[16 + i]);
            epi_gated16(p, bias, bias_up, n, g, u);
        } else {
            epi_finish16(p, bias, brow, n, g);
        }
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = pack_half2(g[2 * i], g[2 * i + 1]);
        emit_piece<kMulti>(p, L, ug, piece, npieces, h, m0, n0, crow, ctma, buf, group_count);
    }
}

// Epilogue of a unit whose tile is cut along K (split-K or stream-K), run by
// the 128 epilogue threads.  This unit's fp32 sum is a partial.  The last unit
// of the tile to finish adds all partials in K order (deterministic) and stores
// C; the others leave their partial in the workspace.  The accumulator stays in
// TMEM until the decision, so the last one takes its own values from TMEM.
// kEpi: the complete sums go through the fused bias + activation stage
// (`bias`, or the row's `brow`) before the store; gated tiles are never cut.
template <bool kPair, bool kMulti, bool kEpi>
__device__ __forceinline__ void cut_tile_epilogue(const KernelParams& p, const SmemLayout& L, const Unit& w,
                                               const UnitGeom& ug, uint32_t taddr, uint32_t tempty, int64_t m0, int64_t n0,
                                               volatile int* flag, volatile int* abort, uint32_t& fix_ph,
                                               bool last_unit, const __half* bias, float brow)
{
    const int lane = threadIdx.x & 31;
    const int row = 32 * ((threadIdx.x >> 5) & 3) + lane;
    constexpr int kRanks = kPair ? 2 : 1;
    const uint32_t rank = kPair ? (cluster_ctarank() & 1u) : 0u;
    const size_t slot_elems = static_cast<size_t>(kBM) * p.BN;   // one CTA's 128 rows of a tile
    int* counter = p.counters + static_cast<size_t>(w.tile) * kRanks + rank;
    const bool lead = threadIdx.x == kEpiLead;
    // Everyone else already in?  Then this unit is last and skips its
    // own write.  (The acquire makes their partials visible.)
    if (lead) *flag = (ld_acquire_gpu(counter) == w.expected - 1) ? 1 : 0;
    named_bar_sync(1, 128);
    int last = *flag;
    if (!last) {
        // Partial layout [column/4][row][4] floats: a warp's 32 rows
        // store 512 contiguous bytes per float4 store.
        float* slot = p.ws + (static_cast<size_t>(w.slot) * kRanks + rank) * slot_elems;
        float* dst = slot + row * 4;
        for (int c0 = 0; c0 < w.bn; c0 += 32) {
            const int cnt = min(2, (w.bn - c0) / 16);
            uint32_t r[32];
            tmem_ld_x16(taddr + c0, r);
            if (cnt > 1) tmem_ld_x16(taddr + c0 + 16, r + 16);
            tmem_wait_ld();
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4)
                if (g4 < 4 * cnt)
                    st_global_v4(dst + static_cast<size_t>(c0 / 4 + g4) * (kBM * 4), __uint_as_float(r[4 * g4]),
                                 __uint_as_float(r[4 * g4 + 1]), __uint_as_float(r[4 * g4 + 2]),
                                 __uint_as_float(r[4 * g4 + 3]));
        }
        // The barrier orders every thread's stores before the leader's
        // device-scope release.
        named_bar_sync(1, 128);
        if (lead) *flag = (atom_add_acq_rel_gpu(counter, 1) == w.expected - 1) ? 1 : 0;
        named_bar_sync(1, 128);
        last = *flag;
    }
    if (!last) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            if (kPair)
                mbar_arrive_cluster(tempty);
            else
                mbar_arrive(tempty);
        }
    } else {
        if (lead) st_relaxed_gpu(counter, 0);   // ready for the next call
        // The other partials come into shared memory by TMA bulk copies of 8 KB
        // pieces (16 columns of one partial), in batches of as many pieces as the
        // landing zone holds, all copies of a batch in flight at once and one
        // wait per batch.  The zone is the 32 KB epilogue buffer, or, for the
        // worker's last unit, the whole stage area: that unit's accumulator is
        // full, so every pipeline stage has been consumed.
        const int others = w.expected - 1;
        if (lane == 0) bulk_wait_group_read<0>();   // TMA stores of C done reading the epilogue buffer
        named_bar_sync(1, 128);
        const uint32_t zone = last_unit ? L.a : L.epi;
        const int cap = static_cast<int>(last_unit ? (L.epi - L.a) / 8192u : kEpiBytes / 8192u);
        const int chunks = w.bn / 16;
        if (others <= 3) {
            // Common case (stream-K and split-K up to four ways): whole chunks per
            // batch, four chunks (64 columns) per TMEM wait, and when the
            // epilogue buffer is free (last unit) and C takes TMA stores, the
            // result goes out through swizzled staging and TMA stores like a
            // whole tile's.
            int per = cap / others;
            if (per >= 4) per &= ~3;
            const int64_t crow = ug.a_row + m0 + 32 * ((threadIdx.x >> 5) & 3);   // this warp's first C row
            // (a TMA store writes a whole 64-column box, so only batches of whole
            // boxes, per >= 4 chunks, may go that way)
            const bool stage_c =
                last_unit && p.c_tma && per >= 4 && (!kMulti || p.gmode != 2 || crow + 32 <= ug.row_lim);
            const int q = (threadIdx.x >> 5) & 3;
            uint32_t gc = 0;   // TMA-store groups this warp issued
            for (int b0 = 0; b0 < chunks; b0 += per) {
                const int nch = min(per, chunks - b0);
                if (lead) {
                    fence_proxy_async_smem();   // the previous batch's generic reads come first
                    const uint32_t fb = bar_fix(L.bars);
                    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nch * others) * 8192u);
                    for (int c = 0; c < nch; ++c)
                        for (int j = 0; j < others; ++j) {
                            const int idx = j < w.seg ? j : j + 1;   // K-order index, own one skipped
                            const size_t sl = static_cast<size_t>(w.slot0 + idx) * kRanks + rank;
                            const float* src =
                                p.ws + sl * slot_elems + static_cast<size_t>(b0 + c) * (4 * kBM * 4);
                            bulk_load(zone + static_cast<uint32_t>(c * others + j) * 8192u, src, 8192, fb);
                        }
                    const bool got = mbar_wait(fb, fix_ph & 1u, abort, p.timeout_ns);
                    if (!got) {
                        raise_abort(p, abort);
                        mbar_wait(fb, fix_ph & 1u, nullptr, kDrainTimeoutNs);   // let the copies land
                    }
                    *flag = got ? 1 : 0;
                }
                fix_ph ^= 1u;
                named_bar_sync(1, 128);
                if (*flag == 0) break;
                for (int g0 = 0; g0 < nch; g0 += 4) {
                    const int gn = min(4, nch - g0);
                    uint32_t buf = 0;
                    if (stage_c) {
                        buf = L.epi + (q * 2 + (gc & 1u)) * kEpiBufBytes;
                        if (lane == 0) bulk_wait_group_read<1>();
                        __syncwarp();
                    }
                    if (others == 1 && gn == 4) {
                        // One other partial (the usual stream-K cut): four chunks per
                        // TMEM wait, every shared-memory load issued before the adds.
                        uint32_t r[64];
#pragma unroll
                        for (int h2 = 0; h2 < 4; ++h2) tmem_ld_x16(taddr + (b0 + g0 + h2) * 16, r + 16 * h2);
                        tmem_wait_ld();
                        const bool own_first = w.seg == 0;
#pragma unroll
                        for (int hp = 0; hp < 4; hp += 2) {   // shared-memory loads two chunks at a time
                            float4 v[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                v[e] = ld_smem_f4(zone + static_cast<uint32_t>(g0 + hp + (e >> 2)) * 8192u + row * 16 +
                                                  (e & 3) * (kBM * 16));
#pragma unroll
                            for (int h1 = 0; h1 < 2; ++h1) {
                                const int h2 = hp + h1;
                                uint32_t h[8];
                                float sv[16];
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    const float o0 = __uint_as_float(r[16 * h2 + 2 * i]);
                                    const float o1 = __uint_as_float(r[16 * h2 + 2 * i + 1]);
                                    const float4& q4 = v[4 * h1 + (i >> 1)];
                                    const float p0 = (i & 1) ? q4.z : q4.x;
                                    const float p1 = (i & 1) ? q4.w : q4.y;
                                    // K order: 0 + first + second, exactly as in the general loop
                                    sv[2 * i] = own_first ? (0.f + o0) + p0 : (0.f + p0) + o0;
                                    sv[2 * i + 1] = own_first ? (0.f + o1) + p1 : (0.f + p1) + o1;
                                }
                                if (kEpi) epi_finish16(p, bias, brow, n0 + (b0 + g0 + h2) * 16, sv);
#pragma unroll
                                for (int i = 0; i < 8; ++i) h[i] = pack_half2(sv[2 * i], sv[2 * i + 1]);
                                if (stage_c) {
                                    const int j0 = h2 * 2;
                                    st_smem_v4(buf + lane * 128 + ((j0 ^ (lane & 7)) << 4),
                                               make_uint4(h[0], h[1], h[2], h[3]));
                                    st_smem_v4(buf + lane * 128 + (((j0 + 1) ^ (lane & 7)) << 4),
                                               make_uint4(h[4], h[5], h[6], h[7]));
                                } else {
                                    store_piece_masked(p, ug.C, ug.row_lim, ug.a_row + m0 + row, n0 + (b0 + g0 + h2) * 16,
                                                       h);
                                }
                            }
                        }
                    } else
                    for (int s0 = 0; s0 < gn; s0 += 2) {   // two chunks (32 columns) per TMEM wait
                        const int sn = min(2, gn - s0);
                        uint32_t r[32];   // this unit's own sums for the two chunks
                        tmem_ld_x16(taddr + (b0 + g0 + s0) * 16, r);
                        if (sn > 1) tmem_ld_x16(taddr + (b0 + g0 + s0 + 1) * 16, r + 16);
                        tmem_wait_ld();
#pragma unroll
                        for (int h1 = 0; h1 < 2; ++h1) {
                            if (h1 >= sn) break;
                            const int c = g0 + s0 + h1;
                            float acc[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[i] = 0.f;
                            for (int j = 0; j < others; ++j) {   // K order, own sum at position seg
                                if (j == w.seg) {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) acc[i] += __uint_as_float(r[16 * h1 + i]);
                                }
                                const uint32_t src =
                                    zone + static_cast<uint32_t>(c * others + j) * 8192u + row * 16;
#pragma unroll
                                for (int g4 = 0; g4 < 4; ++g4) {
                                    const float4 v = ld_smem_f4(src + g4 * (kBM * 16));
                                    acc[4 * g4] += v.x;
                                    acc[4 * g4 + 1] += v.y;
                                    acc[4 * g4 + 2] += v.z;
                                    acc[4 * g4 + 3] += v.w;
                                }
                            }
                            if (w.seg == others) {
#pragma unroll
                                for (int i = 0; i < 16; ++i) acc[i] += __uint_as_float(r[16 * h1 + i]);
                            }
                            if (kEpi) epi_finish16(p, bias, brow, n0 + (b0 + c) * 16, acc);
                            uint32_t h[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) h[i] = pack_half2(acc[2 * i], acc[2 * i + 1]);
                            if (stage_c) {
                                const int j0 = (s0 + h1) * 2;   // 16-byte chunk inside the 128-byte row
                                st_smem_v4(buf + lane * 128 + ((j0 ^ (lane & 7)) << 4),
                                           make_uint4(h[0], h[1], h[2], h[3]));
                                st_smem_v4(buf + lane * 128 + (((j0 + 1) ^ (lane & 7)) << 4),
                                           make_uint4(h[4], h[5], h[6], h[7]));
                            } else {
                                store_piece_masked(p, ug.C, ug.row_lim, ug.a_row + m0 + row, n0 + (b0 + c) * 16, h);
                            }
                        }
                    }
                    if (stage_c) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (crow < ug.row_lim) {
                                const int32_t xn = static_cast<int32_t>(n0 + 16 * (b0 + g0));
                                if (kMulti && p.c_bdim)
                                    tma_store_3d_l2(&p.tmC, buf, xn, static_cast<int32_t>(crow), ug.cz, p.l2_c);
                                else
                                    tma_store_2d_l2(&p.tmC, buf, xn, static_cast<int32_t>(crow), p.l2_c);
                            }
                            bulk_commit_group();
                        }
                        ++gc;
                    }
                }
                named_bar_sync(1, 128);   // the zone is free for the next batch
            }
            if (stage_c && lane == 0) bulk_wait_group_read<0>();   // staging free for the caller's next unit
        } else {
            // Pieces are numbered t = chunk * others + j (j-th other partial of the
            // chunk in K order); a batch holds up to `cap` of them.  Each thread keeps
            // the running sum of the current chunk across batches, adds its own sum
            // (from TMEM) at its K position, and stores the chunk after its last piece.
            const int total = chunks * others;
            float sacc[16];
            for (int t0 = 0; t0 < total; t0 += cap) {
                const int nb = min(cap, total - t0);
                if (lead) {
                    fence_proxy_async_smem();   // the previous batch's generic reads come first
                    const uint32_t fb = bar_fix(L.bars);
                    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nb) * 8192u);
                    for (int u = 0; u < nb; ++u) {
                        const int t = t0 + u, c = t / others, j = t - c * others;
                        const int idx = j < w.seg ? j : j + 1;   // K-order index, own one skipped
                        const size_t sl = static_cast<size_t>(w.slot0 + idx) * kRanks + rank;
                        const float* src = p.ws + sl * slot_elems + static_cast<size_t>(c) * (4 * kBM * 4);
                        bulk_load(zone + static_cast<uint32_t>(u) * 8192u, src, 8192, fb);
                    }
                    const bool got = mbar_wait(fb, fix_ph & 1u, abort, p.timeout_ns);
                    if (!got) {
                        raise_abort(p, abort);
                        mbar_wait(fb, fix_ph & 1u, nullptr, kDrainTimeoutNs);   // let the copies land
                    }
                    *flag = got ? 1 : 0;
                }
                fix_ph ^= 1u;
                named_bar_sync(1, 128);
                if (*flag == 0) break;
                for (int u = 0; u < nb; ++u) {
                    const int t = t0 + u, c = t / others, j = t - c * others;
                    if (j == 0) {
    #pragma unroll
                        for (int i = 0; i < 16; ++i) sacc[i] = 0.f;
                    }
                    // own sum (K index seg) goes before the piece with K index seg + 1;
                    // seg and j are uniform, so the TMEM load is warp-wide
                    if (j == w.seg) add_tmem16(taddr + c * 16, sacc);
                    const uint32_t src = zone + static_cast<uint32_t>(u) * 8192u + row * 16;
    #pragma unroll
                    for (int g4 = 0; g4 < 4; ++g4) {
                        const float4 v = ld_smem_f4(src + g4 * (kBM * 16));
                        sacc[4 * g4] += v.x;
                        sacc[4 * g4 + 1] += v.y;
                        sacc[4 * g4 + 2] += v.z;
                        sacc[4 * g4 + 3] += v.w;
                    }
                    if (j == others - 1) {
                        if (w.seg == others) add_tmem16(taddr + c * 16, sacc);   // own sum is the last in K order
                        if (kEpi) epi_finish16(p, bias, brow, n0 + c * 16, sacc);
                        uint32_t h[8];
    #pragma unroll
                        for (int i = 0; i < 8; ++i) h[i] = pack_half2(sacc[2 * i], sacc[2 * i + 1]);
                        store_piece_masked(p, ug.C, ug.row_lim, ug.a_row + m0 + row, n0 + c * 16, h);
                    }
                }
                named_bar_sync(1, 128);   // the zone is free for the next batch
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            if (kPair)
                mbar_arrive_cluster(tempty);
            else
                mbar_arrive(tempty);
        }
    }
}

// kMulti: batched or grouped launches (gmode != 0); the one-GEMM launch is
// compiled without that geometry.
// kEpi: the fused output stage (bias, activation, gate/up product); built on
// the kMulti geometry, which also runs one-GEMM launches (gmode 0).
template <bool kPair, bool kMulti, bool kEpi = false>
__global__ void __launch_bounds__(kNumThreads, 1) gemm_f16_persistent(const __grid_constant__ KernelParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const SmemLayout L = smem_layout(p, base);
    uint8_t* bars_ptr = smem_raw + (L.bars - raw);
    volatile int* abort = reinterpret_cast<volatile int*>(bars_ptr + kAbortOff);
    volatile int* flag = reinterpret_cast<volatile int*>(bars_ptr + kFlagOff);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars_ptr + kTmemSlotOff);
    volatile int* okflag = reinterpret_cast<volatile int*>(bars_ptr + kOkOff);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool a_tma = p.a_flags & kOpTma, b_tma = p.b_flags & kOpTma;
    const bool a_mn = p.a_flags & kOpMnMajor, b_mn = p.b_flags & kOpMnMajor;
    const bool a_3d = p.a_flags & kOpBox3d, b_3d = p.b_flags & kOpBox3d;
    const bool a_bd = kMulti && p.a_bdim != 0, b_bd = kMulti && p.b_bdim != 0;   // maps with a trailing batch dimension
    static_assert(!kEpi || kMulti, "the fused stage runs on the kMulti single and pair forms");
    const bool gated = kEpi && p.gated != 0;
    const uint32_t crank = kPair ? cluster_ctarank() : 0u;   // rank in the cluster
    const uint32_t rank = crank & 1u;                         // rank in the pair
    const uint32_t lead_rank = crank & ~1u;                   // cluster rank of this pair's leader
    const bool leader = (rank == 0);
    const int cid = static_cast<int>(blockIdx.x >> (kPair ? 1 : 0));
    constexpr int kTileRows = kPair ? 2 * kBM : kBM;
    const int nps = p.stages / kSlots;   // barrier phases in the slot ring

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(bar_full(L.bars, s), p.full_count);
            mbar_init(bar_empty(L.bars, s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull(L.bars, a), 1);
            mbar_init(bar_tempty(L.bars, a), kPair ? 8 : 4);
        }
        mbar_init(bar_drain(L.bars), 1);
        mbar_init(bar_fix(L.bars), 1);
        mbar_init(bar_never(L.bars), 1);
        *abort = 0;
        *flag = 0;
        fence_mbarrier_init();
        if (a_tma) tma_prefetch_desc(&p.tmA);
        if (b_tma) tma_prefetch_desc(&p.tmB);
        if (b_tma && p.tail_split > 1) tma_prefetch_desc(&p.tmB2);
        if (b_tma && gated) tma_prefetch_desc(&p.tmBu);
        if (p.c_tma) {
            tma_prefetch_desc(&p.tmC);
            tma_prefetch_desc(&p.tmC4);
        }
        if (p.k2) {
            tma_prefetch_desc(&p.tmA2k);
            tma_prefetch_desc(&p.tmB2k);
            if (gated) tma_prefetch_desc(&p.tmBu2k);
        }
    }
    if (warp == kMmaWarp) {
        if (kPair) {
            tmem_alloc_pair(L.bars + kTmemSlotOff, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(L.bars + kTmemSlotOff, kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if (kPair)
        cluster_sync_all();   // the peer's barriers are initialised before any remote arrival
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above (barriers, TMEM, descriptor prefetch) may overlap the
    // previous kernel on the stream when this grid was launched as its
    // programmatic dependent; no global memory is touched before that kernel
    // has completed.  The next kernel may then be scheduled as SMs free up (it
    // waits the same way before reading C or the workspace).
    griddep_wait();
    griddep_launch_dependents();

    if (warp < kMmaWarp) {
        // ------------------------------------------------------------ producers
        const int t = threadIdx.x;
        const bool any_masked = !a_tma || !b_tma;
        // The threads that issue TMA copies: with both operands by TMA, one for
        // A' (warp 1) and one for B' (warp 2), so that each copy's issue overlaps
        // the other's (0.3-1 % on the large shapes, e.g. 4096^3 and the
        // 32 x 1024^3 batch); each announces its own bytes on the full barrier,
        // which then expects two arrivals.  With a gathered operand thread 0
        // issues the TMA operand's copies and the producer warps gather the other.
        const int tiss = any_masked ? 0 : kTmaThread;
        const int tiss_b = any_masked ? 0 : kTmaThread + 32;
        const bool do_a = t == tiss, do_b = t == tiss_b;
        if (do_a || do_b || any_masked) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int issued = 0;
            const int nu = units_of_worker(p, cid);
            for (int i = 0; i < nu && ok; ++i) {
                const Unit w = unit_at<kMulti>(p, cid, i);
                const UnitGeom ug = unit_geom<kMulti>(p, w);
                // Columns of one B box: this CTA's share of the unit's B columns.  A
                // gated unit's stage holds BN/2 gate then BN/2 up columns, both at B'
                // column n0: the single form loads both boxes, the pair form's rank 0
                // the gate box and rank 1 the up box.
                const int bcols = (kPair || gated) ? w.bn / 2 : w.bn;
                const int64_t m0 = static_cast<int64_t>(w.m_blk) * kTileRows + rank * kBM;
                const int64_t n0 = gated ? static_cast<int64_t>(w.n_blk) * (p.BN / 2)
                                         : static_cast<int64_t>(w.n_blk) * p.BN + w.n_off + rank * bcols;
                const int64_t arow = ug.a_row + m0;   // A' row of the slot boxes (rows of a group are concatenated)
                // Bytes one stage of this unit brings in: MN-major B comes in
                // 64-column boxes (or one 3-D box of the full stage width),
                // K-major B in one box of the full tile width.  A tail piece
                // narrower than the tile reads B through tmB2, whose box is the
                // piece's width, so it brings only its own columns.
                const bool narrow = w.bn < p.BN;
                const CUtensorMap* tmb = (narrow && !(b_mn && !b_3d)) ? &p.tmB2 : &p.tmB;
                if (kPair && gated && rank == 1) tmb = &p.tmBu;
                const uint32_t b_bytes =
                    (!gated && ((b_mn && !b_3d) || narrow)) ? static_cast<uint32_t>(bcols) * 128u : p.stage_b_bytes;
                const uint32_t tx = kPair ? 2u * (kStageABytes + b_bytes)
                                          : (a_tma ? kStageABytes : 0u) + (b_tma ? b_bytes : 0u);
                for (int kb = w.kb0; kb < w.kb1; kb += kSlots) {
                    const int nk = min(kSlots, w.kb1 - kb);   // K blocks in this barrier phase
                    if (!wait_bar<kPair>(bar_empty(L.bars, stage), phase ^ 1u, abort, p.timeout_ns)) {
                        raise_abort(p, abort);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar_full(L.bars, stage);
                    // The leader (pair form) expects both CTAs' bytes of every slot of
                    // the phase on its own barrier; the peer's copies complete there.
                    if ((a_tma || b_tma) && (!kPair || leader)) {
                        const uint32_t nkb = static_cast<uint32_t>(nk) * (kPair ? 2u : 1u);
                        if (any_masked) {
                            if (do_a) mbar_arrive_expect_tx(fb, tx * static_cast<uint32_t>(nk));
                        } else {
                            if (do_a) mbar_arrive_expect_tx(fb, kStageABytes * nkb);
                            if (do_b) mbar_arrive_expect_tx(fb, b_bytes * nkb);
                        }
                    }
                    // Both K blocks of the phase in one copy per operand (whole K
                    // blocks of a full-width unit): half the TMA instructions, which
                    // the operand feed is sensitive to (131072 x 2048 x 7168: +3 %).
                    // (A gated stage qualifies only in the pair form, where each
                    // CTA's B slot holds one box: the gate or the up columns.)
                    const bool two = p.k2 && nk == 2 && !narrow && kb + 2 <= p.kfull;
                    if (two && (do_a || do_b))
                        load_two_k_blocks<kPair>(p, (kPair && gated && rank == 1) ? &p.tmBu2k : &p.tmB2k,
                                                 L.a + stage * kSlots * kStageABytes,
                                                 L.b + stage * kSlots * p.stage_b_bytes, kb, arow, n0, ug.az, ug.bz,
                                                 a_mn, b_mn, a_bd, b_bd, kPair ? mapa_shared(fb, lead_rank) : fb, do_a,
                                                 do_b);
                    for (int h = 0; h < (two ? 0 : nk); ++h) {
                    const int slot = stage * kSlots + h;
                    const uint32_t sa = L.a + slot * kStageABytes;
                    const uint32_t sb = L.b + slot * p.stage_b_bytes;
                    const int32_t k0 = (kb + h) * kBK;
                    if ((do_a || do_b) && (a_tma || b_tma)) {
                        if (kPair) {
                            const uint32_t fbc = mapa_shared(fb, lead_rank);
                            if (do_a) load_a_slot<true>(p, sa, k0, arow, ug.az, a_mn, a_3d, a_bd, fbc);
                            if (do_b) load_b_slot<true>(p, tmb, sb, k0, n0, ug.bz, bcols, b_mn, b_3d, b_bd, fbc);
                        } else {
                            if (a_tma && do_a) load_a_slot<false>(p, sa, k0, arow, ug.az, a_mn, a_3d, a_bd, fb);
                            if (b_tma && do_b) load_b_slot<false>(p, tmb, sb, k0, n0, ug.bz, bcols, b_mn, b_3d, b_bd, fb);
                            if (b_tma && gated && do_b)
                                load_b_slot<false>(p, &p.tmBu, sb + bcols * 128, k0, n0, ug.bz, bcols, b_mn, b_3d, b_bd,
                                                   fb);
                        }
                    }
                    if (!kPair && any_masked) {
                        if (!a_tma)
                            gather_tile(p, kSpanA, ug.A, p.a_sm, p.a_sk, ug.row_lim, p.K, ug.a_row + m0, k0, kBM, a_mn,
                                        sa, t);
                        if (!b_tma) {
                            // (one inlined gather body for both halves of a gated stage)
#pragma unroll 1
                            for (int hb = 0; hb < (gated ? 2 : 1); ++hb)
                                gather_tile(p, hb ? kSpanBu : kSpanB, hb ? ug.Bu : ug.B, p.b_sn, p.b_sk, p.N, p.K, n0, k0,
                                            bcols, b_mn,
                                            sb + hb * bcols * 128, t);
                        }
                    }
                    }
                    if (!kPair && any_masked) {
                        fence_proxy_async_smem();
                        mbar_arrive(fb);
                    }
                    ++issued;
                    if (++stage == nps) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && (do_a || do_b) && (a_tma || b_tma) && (!kPair || leader)) {
                // Let TMA copies already in flight land before the CTA exits:
                // wait (bounded) on the full barrier of each phase this thread
                // issued recently (one whose other issuer never arrived runs
                // out its bound, by when this thread's own copies have landed).
                const int n = issued < nps ? issued : nps;
                for (int i = 0; i < n; ++i) {
                    if (--stage < 0) {
                        stage = nps - 1;
                        phase ^= 1u;
                    }
                    wait_bar<kPair>(bar_full(L.bars, stage), phase, nullptr, kDrainTimeoutNs);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            bool any = false;
            const uint32_t b_atom_rows = 8192;   // MN-major: one 64-wide atom column over 64 K rows
            const int nu = units_of_worker(p, cid);
            if (p.test_stall && !wait_bar<kPair>(bar_never(L.bars), 0, abort, p.timeout_ns)) {
                raise_abort(p, abort);
                ok = false;
            }
            for (int i = 0; i < nu && ok; ++i) {
                const Unit w = unit_at<kMulti>(p, cid, i);
                if (!wait_bar<kPair>(bar_tempty(L.bars, acc), acc_phase ^ 1u, abort, p.timeout_ns)) {
                    raise_abort(p, abort);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * kAccStride;
                // N field (bits 17-22) of the instruction descriptor: this unit's width
                const uint32_t idesc = (p.idesc & ~(0x3Fu << 17)) | ((static_cast<uint32_t>(w.bn) >> 3) << 17);
                for (int kb = w.kb0; kb < w.kb1; kb += kSlots) {
                    const int nk = min(kSlots, w.kb1 - kb);   // K blocks in this barrier phase
                    if (!wait_bar<kPair>(bar_full(L.bars, stage), phase, abort, p.timeout_ns)) {
                        raise_abort(p, abort);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int h = 0; h < nk; ++h) {
                        const int slot = stage * kSlots + h;
                        const uint32_t sa = L.a + slot * kStageABytes;
                        const uint32_t sb = L.b + slot * p.stage_b_bytes;
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k) {
                            // K-major: the 16-wide K step is 32 bytes inside the
                            // swizzle row.  MN-major: it is 16 K rows of 128 bytes.
                            const uint64_t ad = a_mn ? umma_desc_sw128(sa + k * 2048, 8192, 1024)
                                                     : umma_desc_sw128(sa + k * 32, 16, 1024);
                            const uint64_t bd = b_mn ? umma_desc_sw128(sb + k * 2048, b_atom_rows, 1024)
                                                     : umma_desc_sw128(sb + k * 32, 16, 1024);
                            const uint32_t accum = (kb + h > w.kb0 || k > 0) ? 1u : 0u;
                            if (kPair)
                                umma_f16_pair(d, ad, bd, idesc, accum);
                            else
                                umma_f16(d, ad, bd, idesc, accum);
                        }
                    }
                    any = true;
                    if (kPair)
                        umma_commit_pair_mc(bar_empty(L.bars, stage), 0x3);
                    else
                        umma_commit(bar_empty(L.bars, stage));
                    if (++stage == nps) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (kPair)
                    umma_commit_pair_mc(bar_tfull(L.bars, acc), static_cast<uint16_t>(0x3u << crank));
                else
                    umma_commit(bar_tfull(L.bars, acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok && any) {
                // Drain: wait (bounded) until every MMA issued so far has completed
                // before the accumulator memory is released.
                if (kPair)
                    umma_commit_pair_mc(bar_drain(L.bars), static_cast<uint16_t>(0x1u << crank));
                else
                    umma_commit(bar_drain(L.bars));
                wait_bar<kPair>(bar_drain(L.bars), 0, nullptr, kDrainTimeoutNs);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quarter
        const int row = 32 * q + lane;          // row inside this CTA's 128 rows
        const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t group_count = 0;
        uint32_t fix_ph = 0u;   // bit 0: parity of the next phase of the fixup barrier
        const int nu = units_of_worker(p, cid);
        for (int ui = 0; ui < nu; ++ui) {
            const Unit w = unit_at<kMulti>(p, cid, ui);
            const int64_t m0 = static_cast<int64_t>(w.m_blk) * kTileRows + rank * kBM;
            // first output column (a gated tile has BN/2 of them)
            const int64_t n0 = gated ? static_cast<int64_t>(w.n_blk) * (p.BN / 2)
                                     : static_cast<int64_t>(w.n_blk) * p.BN + w.n_off;
            const int npieces = w.bn / 16;          // 16 accumulator columns per piece
            // One thread waits for the accumulator and tells the other epilogue
            // threads, so that they all leave together on an abort (the named
            // barriers below must see all 128 threads).
            if (threadIdx.x == kEpiLead) {
                const bool ok = wait_bar<kPair>(bar_tfull(L.bars, acc), acc_phase, abort, p.timeout_ns);
                if (!ok) raise_abort(p, abort);
                okflag[acc] = ok ? 1 : 0;
            }
            named_bar_sync(1, 128);
            if (!okflag[acc]) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + lane_off + acc * kAccStride;
            const uint32_t tempty = kPair ? mapa_shared(bar_tempty(L.bars, acc), lead_rank) : bar_tempty(L.bars, acc);
            const UnitGeom ug = unit_geom<kMulti>(p, w);
            // this warp's first row of C, and whether its 32-row boxes go out by TMA
            // store: clipped at the problem's M by the map, except that a box of a
            // group must not spill into the next group's rows
            const int64_t crow = ug.a_row + m0 + 32 * q;
            const bool ctma = p.c_tma && (!kMulti || p.gmode != 2 || crow + 32 <= ug.row_lim);
            // Whole tiles whose 128 rows all go out by TMA store take one
            // 64 x 128 box per 64 columns for the CTA (four times fewer stores
            // than a box per warp; measured 4-5 % faster on the batched 32 x
            // 1024^3 launch, the same elsewhere).  The same for all four
            // epilogue warps.
            const bool cta_store = p.c_tma && (!kMulti || p.gmode != 2 || ug.a_row + m0 + kBM <= ug.row_lim);
            // fused stage: this problem's bias vectors, and the row's own bias
            // value when the bias runs along the kernel view's rows
            const __half* bias = nullptr;
            const __half* bias_up = nullptr;
            float brow = 0.f;
            if (kEpi) {
                const int64_t bo = p.gmode != 0 ? static_cast<int64_t>(w.g) * p.bias_bs : 0;
                if (p.bias) bias = p.bias + bo;
                if (p.bias_up) bias_up = p.bias_up + bo;
                const int64_t mr = ug.a_row + m0 + row;
                if (bias && p.bias_rows && mr < ug.row_lim) brow = __half2float(bias[mr]);
            }
            if (kEpi && w.slot < 0) {
                fused_tile_epilogue<kPair, kMulti>(p, L, ug, bias, bias_up, brow, taddr, tempty, m0, n0,
                                                   gated ? w.bn / 2 : w.bn, gated, crow, ctma, group_count);
            } else if (w.slot < 0) {
                uint32_t buf = 0;
                // Stores of the previous unit may still read the epilogue buffer:
                // the whole-CTA boxes (issued by one thread) cover every warp's part
                // of it, so before this unit stages anything that thread's stores
                // are done reading (each warp tracks its own per-warp boxes).
                if (threadIdx.x == kEpiLead) bulk_wait_group_read<0>();
                if (cta_store && lane == 0) bulk_wait_group_read<0>();
                named_bar_sync(1, 128);
                for (int pc = 0; pc < npieces; pc += 4) {
                    // up to four pieces (64 columns) in flight per TMEM wait
                    const int cnt = min(4, npieces - pc);
                    uint32_t r[64];
#pragma unroll
                    for (int h2 = 0; h2 < 4; ++h2)
                        if (h2 < cnt) tmem_ld_x16(taddr + 16 * (pc + h2), r + 16 * h2);
                    tmem_wait_ld();
                    if (pc + 4 >= npieces) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if (kPair)
                                mbar_arrive_cluster(tempty);
                            else
                                mbar_arrive(tempty);
                        }
                    }
                    if (cta_store) {
                        // the CTA's staging box for these 64 columns: 128 rows, this
                        // warp's 32 of them; one thread stores it once all are staged
                        buf = L.epi + (group_count & 1u) * (4u * kEpiBufBytes) + q * kEpiBufBytes;
                        if (threadIdx.x == kEpiLead) bulk_wait_group_read<1>();   // box free (two stores back)
                        named_bar_sync(1, 128);
                    } else if (ctma || p.c_stage) {
                        buf = L.epi + (q * 2 + (group_count & 1u)) * kEpiBufBytes;
                        if (lane == 0) bulk_wait_group_read<1>();
                        __syncwarp();
                    }
#pragma unroll
                    for (int h2 = 0; h2 < 4; ++h2) {
                        if (h2 >= cnt) break;
                        const int piece = pc + h2;
                        uint32_t h[8];
                        convert16(r + 16 * h2, h);
                        if (cta_store || ctma || p.c_stage) {
                            const int j0 = h2 * 2;        // 16-byte chunk inside the 128-byte row
                            st_smem_v4(buf + lane * 128 + ((j0 ^ (lane & 7)) << 4), make_uint4(h[0], h[1], h[2], h[3]));
                            st_smem_v4(buf + lane * 128 + (((j0 + 1) ^ (lane & 7)) << 4),
                                       make_uint4(h[4], h[5], h[6], h[7]));
                        } else {
                            store_piece_masked(p, ug.C, ug.row_lim, ug.a_row + m0 + row, n0 + 16 * piece, h);
                        }
                    }
                    const int32_t xn = static_cast<int32_t>(n0 + 16 * pc);
                    if (cta_store) {
                        fence_proxy_async_smem();
                        named_bar_sync(1, 128);
                        if (threadIdx.x == kEpiLead) {
                            const int64_t crow0 = ug.a_row + m0;   // (rows past M are clipped by the map)
                            const uint32_t box = L.epi + (group_count & 1u) * (4u * kEpiBufBytes);
                            if (crow0 < ug.row_lim) {
                                if (kMulti && p.c_bdim)
                                    tma_store_3d_l2(&p.tmC4, box, xn, static_cast<int32_t>(crow0), ug.cz, p.l2_c);
                                else
                                    tma_store_2d_l2(&p.tmC4, box, xn, static_cast<int32_t>(crow0), p.l2_c);
                            }
                            bulk_commit_group();
                        }
                        ++group_count;
                    } else if (ctma) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            // (a box wholly below row M, e.g. the second CTA's rows of a
                            // pair tile on the last row, is not stored)
                            if (crow < ug.row_lim) {
                                if (kMulti && p.c_bdim)
                                    tma_store_3d_l2(&p.tmC, buf, xn, static_cast<int32_t>(crow), ug.cz, p.l2_c);
                                else
                                    tma_store_2d_l2(&p.tmC, buf, xn, static_cast<int32_t>(crow), p.l2_c);
                            }
                            bulk_commit_group();
                        }
                        ++group_count;
                    } else if (p.c_stage) {
                        __syncwarp();
                        store_box_rows(p, ug.C, ug.row_lim, buf, crow, n0 + 16 * pc, 16 * cnt);
                        __syncwarp();   // the box is read before the next piece overwrites it
                    }
                }
            } else {
                cut_tile_epilogue<kPair, kMulti, kEpi>(p, L, w, ug, taddr, tempty, m0, n0, flag, abort, fix_ph, ui == nu - 1,
                                                      bias, brow);
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (p.c_tma && lane == 0) bulk_wait_group_all();
    }

    tc_fence_before();
    if (kPair)
        cluster_sync_all();   // the leader's MMAs into this CTA's TMEM and smem are done
    else
        __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        if (kPair)
            tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace gemm_f16_dev
