// Persistent, warp-specialised fp16 GEMM for sm_103a: C = A * B with fp16
// operands, fp32 accumulation in tensor memory (TMEM) and fp16 output.
//
// One CTA per SM walks a list of work units.  A unit is one 128 x BN output
// tile, or, in split-K mode, one K-segment of such a tile.  Roles:
//
//   warps 0-3  producers.  Operands that TMA can address are loaded by one
//              thread with cp.async.bulk.tensor into 128-byte-swizzled shared
//              memory (out-of-range box elements arrive as zeros).  Operands
//              TMA cannot address (unaligned base or pitch, non-unit inner
//              stride) are gathered by all 128 threads with bounds-checked
//              loads, written in the same swizzled layout and published to the
//              tensor core with fence.proxy.async.  Either way the K tail is
//              zero-filled: an index past K is never wrapped back into range.
//   warp 4-7   epilogue.  tcgen05.ld of the fp32 accumulator (warp w reads
//              TMEM lanes 32*(w%4)..+31), convert to fp16, then either stage
//              through swizzled shared memory and TMA-store (clipped to M x N)
//              or store with per-element bounds checks.  In split-K mode the
//              fp32 partial goes to a workspace and the last CTA to finish a
//              tile sums the partials in split order (deterministic).
//   warp 8     TMEM allocation and the MMA issuer (one thread): 4 x
//              tcgen05.mma (K = 16 each) per 64-wide K block into one of two
//              TMEM accumulators, so the epilogue of a tile overlaps the main
//              loop of the next.
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

constexpr int kBM = 128;                 // tile rows = UMMA M
constexpr int kBK = 64;                  // K per stage: one 128-byte swizzle row of fp16
constexpr int kMaxStages = 16;
constexpr int kNumThreads = 288;         // 9 warps
constexpr int kEpiWarp0 = 4;
constexpr int kMmaWarp = 8;
constexpr uint32_t kTmemCols = 512;      // two accumulators of up to 256 columns
constexpr uint32_t kAccStride = 256;
constexpr uint32_t kStageABytes = kBM * kBK * 2;        // 16 KiB
constexpr uint32_t kEpiBufBytes = 32 * 64 * 2;           // one warp's 32 x 64 fp16 box
constexpr uint32_t kEpiBytes = 4 * 2 * kEpiBufBytes;     // 4 warps, double-buffered
constexpr uint32_t kBarrierBytes = 512;
constexpr int kStatusTimeout = 6;

enum : uint32_t { kOpTma = 1u, kOpMnMajor = 2u };

struct KernelParams {
    CUtensorMap tmA;   // A' (K-major: dims {K, M}; MN-major: dims {M, K})
    CUtensorMap tmB;   // B' (K-major: dims {K, N}; MN-major: dims {N, K})
    CUtensorMap tmC;   // C  (dims {N, M}, box 64 x 32)
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
};

struct SmemLayout {
    uint32_t a, b, epi, bars;
};

__device__ __forceinline__ SmemLayout smem_layout(const KernelParams& p, uint32_t base)
{
    SmemLayout s;
    s.a = base;
    s.b = s.a + p.stages * kStageABytes;
    s.epi = s.b + p.stages * p.stage_b_bytes;
    s.bars = s.epi + (p.c_tma ? kEpiBytes : 0u);
    return s;
}

// Barrier block: full[16], empty[16], tmem_full[2], tmem_empty[2], drain,
// then the TMEM base address, the abort flag and a broadcast word.
__device__ __forceinline__ uint32_t bar_full(uint32_t bars, int s) { return bars + 8u * s; }
__device__ __forceinline__ uint32_t bar_empty(uint32_t bars, int s) { return bars + 8u * (kMaxStages + s); }
__device__ __forceinline__ uint32_t bar_tfull(uint32_t bars, int a) { return bars + 8u * (2 * kMaxStages + a); }
__device__ __forceinline__ uint32_t bar_tempty(uint32_t bars, int a) { return bars + 8u * (2 * kMaxStages + 2 + a); }
__device__ __forceinline__ uint32_t bar_drain(uint32_t bars) { return bars + 8u * (2 * kMaxStages + 4); }
constexpr uint32_t kTmemSlotOff = 8u * (2 * kMaxStages + 5);
constexpr uint32_t kAbortOff = kTmemSlotOff + 4;
constexpr uint32_t kFlagOff = kTmemSlotOff + 8;
constexpr uint32_t kOkOff = kTmemSlotOff + 12;   // two words, indexed by accumulator
constexpr uint64_t kDrainTimeoutNs = 10000000ull;

struct Unit {
    int tile, m_blk, n_blk, kb0, kb1;
};

// Work unit -> (tile, K segment).  Units of one tile are consecutive so that
// the split-K partials of a tile sit next to each other.  Tiles are numbered in
// panels of `panel` tile-rows; inside a panel the row index moves fastest, so
// CTAs running at the same time share B columns and a few A row-blocks in L2
// (the grouped program ordering of the Triton page; the C500 review's panel
// rasterisation, section 10).  The ordering is only a locality hint.
__device__ __forceinline__ Unit unit_of(const KernelParams& p, int u)
{
    Unit w;
    w.tile = u / p.splits;
    const int split = u - w.tile * p.splits;
    const int per_panel = p.panel * p.tiles_n;
    const int panel = w.tile / per_panel;
    const int r = w.tile - panel * per_panel;
    const int rows = min(p.panel, p.tiles_m - panel * p.panel);
    w.m_blk = panel * p.panel + r % rows;
    w.n_blk = r / rows;
    w.kb0 = static_cast<int>(static_cast<int64_t>(split) * p.kblocks / p.splits);
    w.kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * p.kblocks / p.splits);
    return w;
}

__device__ __forceinline__ void raise_abort(const KernelParams& p, volatile int* abort)
{
    *abort = 1;
    if (p.status) atomicExch(p.status, kStatusTimeout);
}

// Eight consecutive elements along `step`, starting at element offset `off`;
// the first `nvalid` are loaded, the rest are zero.  Nothing outside the
// caller's bounds is read.
__device__ __forceinline__ uint4 load8(const __half* base, int64_t off, int64_t step, int nvalid)
{
    uint4 r = make_uint4(0u, 0u, 0u, 0u);
    if (nvalid <= 0) return r;
    const uint16_t* q = reinterpret_cast<const uint16_t*>(base) + off;
    if (step == 1 && nvalid >= 8) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(q);
        if ((a & 15u) == 0) return ld_nc_v4(q);
        if ((a & 3u) == 0) {
            r.x = ld_nc_u32(q);
            r.y = ld_nc_u32(q + 2);
            r.z = ld_nc_u32(q + 4);
            r.w = ld_nc_u32(q + 6);
            return r;
        }
    }
    uint32_t v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = (e < nvalid) ? static_cast<uint32_t>(ld_nc_u16(q + e * step)) : 0u;
    r.x = v[0] | (v[1] << 16);
    r.y = v[2] | (v[3] << 16);
    r.z = v[4] | (v[5] << 16);
    r.w = v[6] | (v[7] << 16);
    return r;
}

__device__ __forceinline__ int clamp8(int64_t remaining)
{
    return remaining >= 8 ? 8 : (remaining <= 0 ? 0 : static_cast<int>(remaining));
}

// Gather one operand tile (rows = MN extent `rows_tile`, 64 K columns) into the
// 128B-swizzled layout the UMMA descriptor expects.  K-major: row r (128 B) at
// r*128, its 16-byte chunk j at ((j ^ (r & 7)) << 4).  MN-major: atom column a
// (64 MN elements) at a*8192, K row r at r*128, chunk j swizzled the same way.
__device__ __forceinline__ void gather_tile(const __half* base, int64_t s_mn, int64_t s_k,
                                            int64_t MN, int64_t K, int64_t mn0, int64_t k0,
                                            int rows_tile, bool mn_major, uint32_t dst, int t)
{
    const int chunks = rows_tile * 8;   // 16-byte chunks in the tile
    const int iters = chunks / 128;
    const int atoms = rows_tile / 64;
    for (int i0 = 0; i0 < iters; i0 += 8) {
        uint4 v[8];
        uint32_t addr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i0 + i < iters) {
                const int c = t + 128 * (i0 + i);
                const int j = c & 7;
                int64_t mn, k, step;
                int nvalid;
                if (!mn_major) {
                    const int r = c >> 3;
                    mn = mn0 + r;
                    k = k0 + 8 * j;
                    nvalid = (mn < MN) ? clamp8(K - k) : 0;
                    step = s_k;
                    addr[i] = dst + r * 128 + ((j ^ (r & 7)) << 4);
                } else {
                    const int a = (c >> 3) % atoms;
                    const int r = (c >> 3) / atoms;
                    mn = mn0 + 64 * a + 8 * j;
                    k = k0 + r;
                    nvalid = (k < K) ? clamp8(MN - mn) : 0;
                    step = s_mn;
                    addr[i] = dst + a * 8192 + r * 128 + ((j ^ (r & 7)) << 4);
                }
                v[i] = (nvalid > 0) ? load8(base, mn * s_mn + k * s_k, step, nvalid)
                                    : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i0 + i < iters) st_smem_v4(addr[i], v[i]);
    }
}

__device__ __forceinline__ uint16_t half_bits(const uint32_t* h, int c)
{
    return static_cast<uint16_t>(h[c >> 1] >> ((c & 1) * 16));
}

// Store `cols` (<= 64) fp16 values of output row m, columns n.., with bounds
// checks on both m and every column.
__device__ __forceinline__ void store_row_masked(const KernelParams& p, int64_t m, int64_t n, int cols,
                                                 const uint32_t* h)
{
    if (m >= p.M) return;
    uint16_t* row = reinterpret_cast<uint16_t*>(p.C) + m * p.c_sm;
    if (p.c_sn == 1) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (8 * j < cols) {
                const int64_t nn = n + 8 * j;
                uint16_t* q = row + nn;
                if (nn + 8 <= p.N && (reinterpret_cast<uintptr_t>(q) & 15u) == 0) {
                    *reinterpret_cast<uint4*>(q) =
                        make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (nn + e < p.N) q[e] = half_bits(h, 8 * j + e);
                }
            }
        }
    } else {
#pragma unroll
        for (int c = 0; c < 64; ++c)
            if (c < cols && n + c < p.N) row[(n + c) * p.c_sn] = half_bits(h, c);
    }
}

// Load up to 64 accumulator columns [col0, col0+cols) of this thread's lane.
__device__ __forceinline__ void tmem_load_group(uint32_t taddr, int cols, uint32_t* r)
{
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (16 * i < cols) tmem_ld_x16(taddr + 16 * i, r + 16 * i);
    tmem_wait_ld();
}

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

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(bar_full(L.bars, s), p.full_count);
            mbar_init(bar_empty(L.bars, s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull(L.bars, a), 1);
            mbar_init(bar_tempty(L.bars, a), 4);
        }
        mbar_init(bar_drain(L.bars), 1);
        *abort = 0;
        *flag = 0;
        fence_mbarrier_init();
        if (a_tma) tma_prefetch_desc(&p.tmA);
        if (b_tma) tma_prefetch_desc(&p.tmB);
        if (p.c_tma) tma_prefetch_desc(&p.tmC);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(L.bars + kTmemSlotOff, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp < 4) {
        // ------------------------------------------------------------ producers
        const int t = threadIdx.x;
        const bool any_masked = !a_tma || !b_tma;
        if (t == 0 || any_masked) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int issued = 0;
            for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
                const Unit w = unit_of(p, u);
                const int64_t m0 = static_cast<int64_t>(w.m_blk) * kBM;
                const int64_t n0 = static_cast<int64_t>(w.n_blk) * p.BN;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_wait(bar_empty(L.bars, stage), phase ^ 1u, abort, p.timeout_ns)) {
                        raise_abort(p, abort);
                        ok = false;
                        break;
                    }
                    const uint32_t sa = L.a + stage * kStageABytes;
                    const uint32_t sb = L.b + stage * p.stage_b_bytes;
                    const uint32_t fb = bar_full(L.bars, stage);
                    const int32_t k0 = kb * kBK;
                    if (t == 0 && (a_tma || b_tma)) {
                        mbar_arrive_expect_tx(fb, p.tx_bytes);
                        if (a_tma) {
                            if (!a_mn) {
                                tma_load_2d(sa, &p.tmA, k0, static_cast<int32_t>(m0), fb);
                            } else {
                                tma_load_2d(sa, &p.tmA, static_cast<int32_t>(m0), k0, fb);
                                tma_load_2d(sa + 8192, &p.tmA, static_cast<int32_t>(m0 + 64), k0, fb);
                            }
                        }
                        if (b_tma) {
                            if (!b_mn) {
                                tma_load_2d(sb, &p.tmB, k0, static_cast<int32_t>(n0), fb);
                            } else {
                                for (int j = 0; j < p.BN / 64; ++j)
                                    tma_load_2d(sb + j * 8192, &p.tmB, static_cast<int32_t>(n0 + 64 * j), k0, fb);
                            }
                        }
                    }
                    if (any_masked) {
                        if (!a_tma)
                            gather_tile(p.A, p.a_sm, p.a_sk, p.M, p.K, m0, k0, kBM, a_mn, sa, t);
                        if (!b_tma)
                            gather_tile(p.B, p.b_sn, p.b_sk, p.N, p.K, n0, k0, p.BN, b_mn, sb, t);
                        fence_proxy_async_smem();
                        mbar_arrive(fb);
                    }
                    ++issued;
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && t == 0 && (a_tma || b_tma)) {
                // Let TMA copies already in flight land before the CTA exits:
                // wait (bounded) on the full barrier of each recently issued stage.
                const int n = issued < p.stages ? issued : p.stages;
                for (int i = 0; i < n; ++i) {
                    if (--stage < 0) {
                        stage = p.stages - 1;
                        phase ^= 1u;
                    }
                    mbar_wait(bar_full(L.bars, stage), phase, nullptr, kDrainTimeoutNs);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            bool any = false;
            for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
                const Unit w = unit_of(p, u);
                if (!mbar_wait(bar_tempty(L.bars, acc), acc_phase ^ 1u, abort, p.timeout_ns)) {
                    raise_abort(p, abort);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * kAccStride;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_wait(bar_full(L.bars, stage), phase, abort, p.timeout_ns)) {
                        raise_abort(p, abort);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = L.a + stage * kStageABytes;
                    const uint32_t sb = L.b + stage * p.stage_b_bytes;
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        // K-major: the 16-wide K step is 32 bytes inside the
                        // swizzle row.  MN-major: it is 16 K rows of 128 bytes.
                        const uint64_t ad = a_mn ? umma_desc_sw128(sa + k * 2048, 8192, 1024)
                                                 : umma_desc_sw128(sa + k * 32, 16, 1024);
                        const uint64_t bd = b_mn ? umma_desc_sw128(sb + k * 2048, 8192, 1024)
                                                 : umma_desc_sw128(sb + k * 32, 16, 1024);
                        umma_f16(d, ad, bd, p.idesc, (kb > w.kb0 || k > 0) ? 1u : 0u);
                    }
                    any = true;
                    umma_commit(bar_empty(L.bars, stage));
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(bar_tfull(L.bars, acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok && any) {
                // Drain: wait (bounded) until every MMA issued so far has completed
                // before the accumulator memory is released.
                umma_commit(bar_drain(L.bars));
                mbar_wait(bar_drain(L.bars), 0, nullptr, kDrainTimeoutNs);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quarter
        const int row = 32 * q + lane;          // row inside the tile
        const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t group_count = 0;
        const int ngroups = (p.BN + 63) / 64;
        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
            const Unit w = unit_of(p, u);
            const int64_t m0 = static_cast<int64_t>(w.m_blk) * kBM;
            const int64_t n0 = static_cast<int64_t>(w.n_blk) * p.BN;
            // One thread waits for the accumulator and tells the other epilogue
            // threads, so that they all leave together on an abort (the named
            // barriers below must see all 128 threads).
            if (threadIdx.x == kEpiWarp0 * 32) {
                const bool ok = mbar_wait(bar_tfull(L.bars, acc), acc_phase, abort, p.timeout_ns);
                if (!ok) raise_abort(p, abort);
                okflag[acc] = ok ? 1 : 0;
            }
            named_bar_sync(1, 128);
            if (!okflag[acc]) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + lane_off + acc * kAccStride;
            if (p.splits == 1) {
                for (int g = 0; g < ngroups; ++g) {
                    const int cols = min(64, p.BN - 64 * g);
                    uint32_t r[64];
                    tmem_load_group(taddr + 64 * g, cols, r);
                    if (g == ngroups - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_tempty(L.bars, acc));
                    }
                    uint32_t h[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        h[i] = pack_half2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                    if (p.c_tma) {
                        const uint32_t buf = L.epi + (q * 2 + (group_count & 1u)) * kEpiBufBytes;
                        if (lane == 0) bulk_wait_group_read<1>();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            st_smem_v4(buf + lane * 128 + ((j ^ (lane & 7)) << 4),
                                       make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]));
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&p.tmC, buf, static_cast<int32_t>(n0 + 64 * g),
                                         static_cast<int32_t>(m0 + 32 * q));
                            bulk_commit_group();
                        }
                        ++group_count;
                    } else {
                        store_row_masked(p, m0 + row, n0 + 64 * g, cols, h);
                    }
                }
            } else {
                // Split-K: write this segment's fp32 partial, column-major inside
                // the unit slot so that a warp's 32 rows form one 128-byte line.
                float* slot = p.ws + static_cast<size_t>(u) * (kBM * p.BN);
                for (int g = 0; g < ngroups; ++g) {
                    const int cols = min(64, p.BN - 64 * g);
                    uint32_t r[64];
                    tmem_load_group(taddr + 64 * g, cols, r);
                    if (g == ngroups - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_tempty(L.bars, acc));
                    }
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (c < cols) slot[(64 * g + c) * kBM + row] = __uint_as_float(r[c]);
                }
                __threadfence();
                named_bar_sync(1, 128);
                if (threadIdx.x == kEpiWarp0 * 32) {
                    const int old = atomicAdd(p.counters + w.tile, 1);
                    const int last = (old == p.splits - 1) ? 1 : 0;
                    if (last) p.counters[w.tile] = 0;   // ready for the next call
                    *flag = last;
                }
                named_bar_sync(1, 128);
                if (*flag) {
                    __threadfence();
                    const float* tb = p.ws + static_cast<size_t>(w.tile) * p.splits * (kBM * p.BN);
                    for (int g = 0; g < ngroups; ++g) {
                        const int cols = min(64, p.BN - 64 * g);
                        float s[64];
#pragma unroll
                        for (int c = 0; c < 64; ++c) s[c] = 0.f;
                        for (int sp = 0; sp < p.splits; ++sp) {
                            const float* src = tb + static_cast<size_t>(sp) * (kBM * p.BN) + (64 * g) * kBM + row;
#pragma unroll
                            for (int c = 0; c < 64; ++c)
                                if (c < cols) s[c] += ld_cg_f32(src + c * kBM);
                        }
                        uint32_t h[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) h[i] = pack_half2(s[2 * i], s[2 * i + 1]);
                        store_row_masked(p, m0 + row, n0 + 64 * g, cols, h);
                    }
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (p.c_tma && lane == 0) bulk_wait_group_all();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace gemm_f16_dev
