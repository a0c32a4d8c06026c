// Repack of an operand that TMA cannot address into a dense, 16-byte-aligned
// copy, so that the GEMM can run its TMA path on the copy.
//
// The pages give two ways to meet a tile boundary that the data does not
// respect: masks, or padding with the extra storage and traffic accounted for
// (AI-infra knowledge base "Matrix multiplication and memory-access
// optimisation", section 05; the mask side is the Triton GEMM page's
// boundary handling).  The in-kernel gather is the mask form.  It re-reads and
// re-aligns an operand once per tile that uses it, which costs more than one
// aligned copy once the operand is reused across many tiles.  This kernel is
// the padding form: it reads the view once, realigns every row, and writes rows
// whose pitch is a multiple of 8 elements (16 bytes), zero-filling the padding.
// It is HBM-bound: 2 bytes read and 2 written per element.
#pragma once

#include <cuda_fp16.h>

#include "gemm_kernel.cuh"

namespace gemm_f16_dev {

constexpr int kRepackThreads = 256;
constexpr int kRepackUnroll = 4;   // 16-byte output chunks a lane has in flight

struct RepackArgs {
    const __half* src;   // element (b, r, c) at src + b*s_b + r*s_r + c*s_c
    int64_t s_r, s_c, s_b;
    __half* dst;         // element (b, r, c) at dst + b*dst_bs + r*pitch + c
    int64_t pitch, dst_bs;
    int64_t rows, cols, batch;
};

// Up to three copies (A', B', the up projection) in one launch: their work
// items are numbered one copy after the other.
struct RepackBatch {
    RepackArgs c[3];
    int n;
};

__host__ __device__ inline int64_t repack_items(const RepackArgs& a)
{
    const int64_t seg = 32 * kRepackUnroll;
    return a.rows * a.batch * ((a.pitch / 8 + seg - 1) / seg);
}

// 8 fp16 values of the 16 bytes at byte offset sh (even) of the 32-byte pair
// w0:w1; the offset is the same for the whole row, so the branch is uniform
// across the warp.
__device__ __forceinline__ uint4 repack_shift(const uint4& w0, const uint4& w1, uint32_t sh)
{
    return sh == 0 ? w0 : funnel16(w0, w1, sh);
}

// Work items are (row, segment of 32 * kRepackUnroll output chunks), one warp
// each, grid-stride over batch * rows * segments, so that a long row does not
// serialise one warp on several memory round trips.  Unit column stride: the
// lane loads the aligned 16-byte source words that hold its output chunk's
// valid elements (never a word without one, so no load leaves the view's
// pages), shifts them into place and stores the chunk.  Other strides: element
// by element.
__global__ void __launch_bounds__(kRepackThreads) repack_rows(const __grid_constant__ RepackBatch batch)
{
    // (as a programmatic dependent: the previous kernel, which may still read
    // this buffer or write the source, has completed)
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kRepackThreads / 32);
    constexpr int64_t kSeg = 32 * kRepackUnroll;
    const int64_t n0 = batch.n > 0 ? repack_items(batch.c[0]) : 0;
    const int64_t n1 = batch.n > 1 ? repack_items(batch.c[1]) : 0;
    const int64_t total = n0 + n1 + (batch.n > 2 ? repack_items(batch.c[2]) : 0);
    for (int64_t qq = static_cast<int64_t>(blockIdx.x) * (kRepackThreads / 32) + (threadIdx.x >> 5); qq < total;
         qq += warps) {
        const int ci = qq < n0 ? 0 : (qq < n0 + n1 ? 1 : 2);
        const RepackArgs& a = batch.c[ci];
        const int64_t q = qq - (ci == 0 ? 0 : (ci == 1 ? n0 : n0 + n1));
        const int64_t chunks = a.pitch / 8;
        const int64_t segs = (chunks + kSeg - 1) / kSeg;
        const int64_t row = q / segs, seg = q - row * segs;
        const int64_t b = row / a.rows, r = row - b * a.rows;
        const __half* srow = a.src + b * a.s_b + r * a.s_r;
        uint4* drow = reinterpret_cast<uint4*>(a.dst + b * a.dst_bs + r * a.pitch);
        const int64_t j0 = seg * kSeg + lane;
        if (a.s_c == 1) {
            const uintptr_t addr = reinterpret_cast<uintptr_t>(srow);
            const uint32_t sh = static_cast<uint32_t>(addr & 15u);
            const uint4* w = reinterpret_cast<const uint4*>(addr - sh);
            uint4 w0[kRepackUnroll], w1[kRepackUnroll];
            int nv[kRepackUnroll];
#pragma unroll
            for (int u = 0; u < kRepackUnroll; ++u) {
                const int64_t j = j0 + 32 * u;
                const int64_t left = a.cols - 8 * j;
                nv[u] = j < chunks ? (left >= 8 ? 8 : (left <= 0 ? 0 : static_cast<int>(left))) : 0;
                w0[u] = w1[u] = make_uint4(0u, 0u, 0u, 0u);
                if (nv[u] > 0) w0[u] = ld_nc_v4(w + j);
                if (nv[u] > 0 && sh + 2u * static_cast<uint32_t>(nv[u]) > 16u) w1[u] = ld_nc_v4(w + j + 1);
            }
#pragma unroll
            for (int u = 0; u < kRepackUnroll; ++u) {
                const int64_t j = j0 + 32 * u;
                if (j >= chunks) break;
                uint4 c = repack_shift(w0[u], w1[u], sh);
                if (nv[u] < 8) c = keep_first(c, nv[u]);
                drow[j] = c;
            }
        } else {
            uint16_t* d = reinterpret_cast<uint16_t*>(drow);
            const uint16_t* s = reinterpret_cast<const uint16_t*>(srow);
            for (int64_t c = 8 * (seg * kSeg) + lane; c < a.pitch && c < 8 * (seg + 1) * kSeg; c += 32)
                d[c] = c < a.cols ? ld_nc_u16(s + c * a.s_c) : uint16_t(0);
        }
    }
}

}  // namespace gemm_f16_dev

namespace gemm_f16_dev {

// The reverse copy, for a C that TMA cannot store (a pitch that is not a
// multiple of 8 elements, or an unaligned base): the GEMM stores its tiles by
// TMA into an aligned buffer (rows `spitch` elements apart, a multiple of 8),
// and this kernel moves the M x N view into C.  Only the view's elements are
// written: C's pitch padding is never touched.  Aligned 16-byte loads; each
// lane then assembles the aligned 16-byte chunk of the destination row that
// its data falls in (a funnel shift of its own and the previous lane's
// bytes), so whole chunks go out as 16-byte stores and only the two ragged
// ends of a row segment take 2-byte stores.  HBM-bound: 2 bytes read and 2
// written per element.
struct UnpackArgs {
    const __half* src;   // element (b, r, c) at src + b*sbs + r*spitch + c; 16-byte-aligned rows
    int64_t spitch, sbs;
    __half* dst;         // element (b, r, c) at dst + b*dbs + r*ldc + c
    int64_t ldc, dbs;
    int64_t rows, cols, batch;
};

constexpr int kUnpackSeg = 256;   // elements of a row one warp moves per work item
constexpr int kUnpackUnroll = 4;  // work items a warp has in flight (their loads issued together)

__host__ __device__ inline int64_t unpack_items(const UnpackArgs& a)
{
    return a.batch * a.rows * ((a.cols + kUnpackSeg - 1) / kUnpackSeg);
}

// Store the halfwords [lo, hi) of a 16-byte chunk (byte offsets lo, hi even).
__device__ __forceinline__ void store_chunk_part(uint16_t* chunk, const uint4& v, uint32_t lo, uint32_t hi)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (uint32_t i = 0; i < 8; ++i)
        if (2 * i >= lo && 2 * i < hi) chunk[i] = static_cast<uint16_t>(w[i >> 1] >> ((i & 1) * 16));
}

// One work item (a segment of up to 256 elements of one row) whose source
// chunk `cur` this lane has already loaded: realign and store.
__device__ __forceinline__ void unpack_store(uint16_t* d, int64_t nvalid, const uint4& cur, int lane)
{
    const uintptr_t D = reinterpret_cast<uintptr_t>(d);
    const uint32_t o = static_cast<uint32_t>(D & 15u);      // even
    uint16_t* A = reinterpret_cast<uint16_t*>(D - o);       // aligned chunk 0
    const uint32_t vbytes = 2u * static_cast<uint32_t>(nvalid);   // valid bytes from D
    uint4 prev;
    prev.x = __shfl_up_sync(0xffffffffu, cur.x, 1);
    prev.y = __shfl_up_sync(0xffffffffu, cur.y, 1);
    prev.z = __shfl_up_sync(0xffffffffu, cur.z, 1);
    prev.w = __shfl_up_sync(0xffffffffu, cur.w, 1);
    // chunk `lane`: destination bytes [16*lane, 16*lane + 16) from A, i.e.
    // bytes [16 - o, 32 - o) of prev:cur (o = 0: cur itself)
    const uint4 chunk = o == 0 ? cur : funnel16(prev, cur, 16u - o);
    // valid bytes of this chunk, relative to A: [o, o + vbytes)
    const uint32_t lo = 16u * lane, hi = lo + 16u;
    const uint32_t vlo = o > lo ? o : lo, vhi = (o + vbytes) < hi ? (o + vbytes) : hi;
    if (vlo < vhi) {
        uint16_t* cp = A + 8 * lane;
        if (vlo == lo && vhi == hi)
            *reinterpret_cast<uint4*>(cp) = chunk;
        else
            store_chunk_part(cp, chunk, vlo - lo, vhi - lo);
    }
    // chunk 32: the last lane's final o bytes when the segment is full
    const uint4 last = make_uint4(__shfl_sync(0xffffffffu, cur.x, 31), __shfl_sync(0xffffffffu, cur.y, 31),
                                  __shfl_sync(0xffffffffu, cur.z, 31), __shfl_sync(0xffffffffu, cur.w, 31));
    if (lane == 0 && o != 0 && o + vbytes > 512u) {
        const uint4 tail = funnel16(last, make_uint4(0u, 0u, 0u, 0u), 16u - o);
        store_chunk_part(A + 8 * 32, tail, 0u, o + vbytes - 512u);
    }
}

__global__ void __launch_bounds__(kRepackThreads) unpack_rows(const __grid_constant__ UnpackArgs a)
{
    // (as a programmatic dependent of the GEMM: its TMA stores are complete
    // and visible once this returns)
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kRepackThreads / 32);
    const int64_t segs = (a.cols + kUnpackSeg - 1) / kUnpackSeg;
    const int64_t total = unpack_items(a);
    // A warp takes kUnpackUnroll consecutive items per pass: every load first,
    // then the realigned stores, so several loads are in flight per lane.
    for (int64_t q0 = (static_cast<int64_t>(blockIdx.x) * (kRepackThreads / 32) + (threadIdx.x >> 5)) * kUnpackUnroll;
         q0 < total; q0 += warps * kUnpackUnroll) {
        uint4 cur[kUnpackUnroll];
        uint16_t* d[kUnpackUnroll];
        int64_t nv[kUnpackUnroll];
#pragma unroll
        for (int u = 0; u < kUnpackUnroll; ++u) {
            const int64_t qq = q0 + u;
            nv[u] = 0;
            d[u] = nullptr;
            cur[u] = make_uint4(0u, 0u, 0u, 0u);
            if (qq < total) {
                const int64_t row = qq / segs, seg = qq - row * segs;
                const int64_t b = row / a.rows, r = row - b * a.rows;
                const int64_t c0 = seg * kUnpackSeg;
                nv[u] = a.cols - c0 < kUnpackSeg ? a.cols - c0 : kUnpackSeg;
                d[u] = reinterpret_cast<uint16_t*>(a.dst + b * a.dbs + r * a.ldc + c0);
                // (the load stays inside the source row's padded pitch)
                if (8 * lane < nv[u]) cur[u] = ld_nc_v4(a.src + b * a.sbs + r * a.spitch + c0 + 8 * lane);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnpackUnroll; ++u)
            if (q0 + u < total) unpack_store(d[u], nv[u], cur[u], lane);   // (uniform across the warp)
    }
}

}  // namespace gemm_f16_dev
