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
constexpr int kCopyUnroll = 4;                   // 16-byte destination chunks a lane has in flight per item
constexpr int kCopySeg = 32 * kCopyUnroll;       // destination chunks of one work item (2 KB)
constexpr int kRepackBlocksPerSm = 4;            // resident blocks (the register budget of __launch_bounds__)
constexpr int kUnpackBlocksPerSm = 4;

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

// Work items of a copy: (row, segment of kCopySeg destination chunks).
__host__ __device__ inline int64_t repack_segs(const RepackArgs& a) { return (a.pitch / 8 + kCopySeg - 1) / kCopySeg; }
__host__ __device__ inline int64_t repack_items(const RepackArgs& a) { return a.rows * a.batch * repack_segs(a); }

// One work item of a row copy with realignment: destination bytes [od, od +
// wlen) relative to the aligned chunk base of the row's destination (od = its
// offset in a 16-byte chunk) receive the row's source bytes [0, len) and,
// past them, zeros (kZero; wlen = len otherwise).  The lane handles the
// destination chunks k = seg * kCopySeg + 32 u + lane.  Destination chunk k
// holds the bytes of two consecutive aligned source chunks, k and its
// neighbour (k + 1 when the source's offset in its chunk is at least the
// destination's, k - 1 otherwise), from a byte offset that is the same for the
// whole row.  The lane loads source chunk k (only chunks with at least one
// byte of the row, so no load leaves the row's pages) and takes the neighbour
// from the next or previous lane with one shuffle per word; at the item's
// edge the lane on the wrap-around side takes it from its own extra load.  It
// shifts the pair into place and stores whole chunks with one 16-byte store;
// only a ragged first or last chunk of a row takes 2-byte stores.  Every load
// is issued before the first store.
template <bool kZero>
__device__ __forceinline__ void copy_row_segment(const __half* src, __half* dst, int64_t len, int64_t wlen,
                                                 int64_t seg, int lane)
{
    const uintptr_t sa = reinterpret_cast<uintptr_t>(src), da = reinterpret_cast<uintptr_t>(dst);
    const int os = static_cast<int>(sa & 15u), od = static_cast<int>(da & 15u);
    const uint4* S = reinterpret_cast<const uint4*>(sa - os);
    uint4* D = reinterpret_cast<uint4*>(da - od);
    // destination chunk k = source bytes [16k + t, 16k + t + 16) relative to S
    const int t = os - od;
    const bool up = t >= 0;   // pair (k, k + 1) from byte t; else (k - 1, k) from byte 16 + t
    const uint32_t sh = static_cast<uint32_t>(up ? t : 16 + t);
    // (chunk counts of a row fit 32 bits: a row holds fewer than 2^31 elements)
    const int64_t vend = od + len, wend = od + wlen;   // copied / written bytes end, relative to D
    const uint32_t nsrc = static_cast<uint32_t>((os + len + 15) >> 4);   // source chunks holding bytes of the row
    const uint32_t nch = static_cast<uint32_t>((wend + 15) >> 4);        // destination chunks written
    const uint32_t kw1 = static_cast<uint32_t>(wend >> 4);               // end of the whole destination chunks
    const uint32_t kv = static_cast<uint32_t>(vend >> 4);                // chunk holding the end of the copied bytes
    const int vrem = static_cast<int>(vend & 15);
    const uint32_t kb = static_cast<uint32_t>(seg) * kCopySeg, k0 = kb + static_cast<uint32_t>(lane);
    uint4 w[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const uint32_t k = k0 + 32u * u;
        w[u] = k < nsrc ? ld_nc_v4(S + k) : make_uint4(0u, 0u, 0u, 0u);
    }
    // the neighbour beyond the item: chunk kb + kCopySeg for lane 31 (up), kb - 1 for lane 0
    uint4 extra = make_uint4(0u, 0u, 0u, 0u);
    if (sh != 0 && lane == (up ? 31 : 0)) {
        const uint32_t kx = up ? kb + kCopySeg : kb - 1u;   // (kb - 1 wraps to 2^32 - 1 for kb = 0: not < nsrc)
        if (kx < nsrc) extra = ld_nc_v4(S + kx);
    }
    const int from = up ? ((lane + 1) & 31) : ((lane + 31) & 31);
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const uint32_t k = k0 + 32u * u;
        uint4 c = w[u];
        if (sh != 0) {
            // the wrap-around lane reads the chunk 32 lanes on: the first lane's
            // next chunk (up) or the last lane's previous one
            uint4 give = w[u];
            if (up && lane == 0 && u + 1 < kCopyUnroll) give = w[u + 1];
            if (!up && lane == 31 && u > 0) give = w[u - 1];
            uint4 nb;
            nb.x = __shfl_sync(0xffffffffu, give.x, from);
            nb.y = __shfl_sync(0xffffffffu, give.y, from);
            nb.z = __shfl_sync(0xffffffffu, give.z, from);
            nb.w = __shfl_sync(0xffffffffu, give.w, from);
            if (up && lane == 31 && u + 1 == kCopyUnroll) nb = extra;
            if (!up && lane == 0 && u == 0) nb = extra;
            c = up ? funnel16(w[u], nb, sh) : funnel16(nb, w[u], sh);
        }
        if (k >= nch) continue;
        if (kZero && k >= kv) c = keep_first(c, k == kv ? vrem / 2 : 0);
        if ((k > 0 || od == 0) && k < kw1) {
            D[k] = c;
        } else {   // the row's ragged first or last chunk: bytes [od, 16) of chunk 0, [0, wend - 16k) of the last
            const uint32_t wd[4] = {c.x, c.y, c.z, c.w};
            uint16_t* cp = reinterpret_cast<uint16_t*>(D + k);
            const int b0 = k == 0 ? od : 0, b1 = k < kw1 ? 16 : static_cast<int>(wend & 15);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (2 * i >= b0 && 2 * i < b1) cp[i] = static_cast<uint16_t>(wd[i >> 1] >> ((i & 1) * 16));
        }
    }
}

// Work items go to the warps round-robin (item q to warp q mod warps), so
// the warps in flight at any time cover one contiguous stretch of the rows.
__device__ __forceinline__ int64_t warp_index() { return static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5); }
__device__ __forceinline__ int64_t warp_count() { return static_cast<int64_t>(gridDim.x) * (blockDim.x / 32); }

// Item q of one copy.  Unit column stride: copy_row_segment (destination
// rows aligned, zero-filled from the view's columns to the pitch); other
// column strides element by element.
__device__ __forceinline__ void repack_item(const RepackArgs& a, int64_t q, int lane)
{
    const int64_t segs = repack_segs(a);
    const int64_t row = q / segs, seg = q - row * segs;
    const int64_t b = row / a.rows, r = row - b * a.rows;
    const __half* srow = a.src + b * a.s_b + r * a.s_r;
    __half* drow = a.dst + b * a.dst_bs + r * a.pitch;
    if (a.s_c == 1) {
        copy_row_segment<true>(srow, drow, 2 * a.cols, 2 * a.pitch, seg, lane);
    } else {
        uint16_t* d = reinterpret_cast<uint16_t*>(drow);
        const uint16_t* sp = reinterpret_cast<const uint16_t*>(srow);
        const int64_t c1 = 8 * (seg + 1) * kCopySeg < a.pitch ? 8 * (seg + 1) * kCopySeg : a.pitch;
        for (int64_t c = 8 * seg * kCopySeg + lane; c < c1; c += 32)
            d[c] = c < a.cols ? ld_nc_u16(sp + c * a.s_c) : uint16_t(0);
    }
}

__global__ void __launch_bounds__(kRepackThreads, kRepackBlocksPerSm) repack_rows(const __grid_constant__ RepackBatch batch)
{
    // (as a programmatic dependent: the previous kernel, which may still read
    // this buffer or write the source, has completed)
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t n0 = batch.n > 0 ? repack_items(batch.c[0]) : 0;
    const int64_t n1 = batch.n > 1 ? repack_items(batch.c[1]) : 0;
    const int64_t total = n0 + n1 + (batch.n > 2 ? repack_items(batch.c[2]) : 0);
    // (the copies' items are numbered one copy after the other)
    for (int64_t q = warp_index(); q < total; q += warp_count()) {
        const int ci = q < n0 ? 0 : (q < n0 + n1 ? 1 : 2);
        repack_item(batch.c[ci], q - (ci == 0 ? 0 : (ci == 1 ? n0 : n0 + n1)), lane);
    }
}

}  // namespace gemm_f16_dev

namespace gemm_f16_dev {

// The reverse copy, for a C that TMA cannot store (a pitch that is not a
// multiple of 8 elements, or an unaligned base): the GEMM stores its tiles by
// TMA into an aligned buffer (rows `spitch` elements apart, a multiple of 8),
// and this kernel moves the M x N view into C.  Only the view's elements are
// written: C's pitch padding is never touched.  copy_row_segment with aligned
// source rows: whole destination chunks go out as 16-byte stores and only the
// two ragged ends of a row take 2-byte stores.  HBM-bound: 2 bytes read and 2
// written per element.
struct UnpackArgs {
    const __half* src;   // element (b, r, c) at src + b*sbs + r*spitch + c; 16-byte-aligned rows
    int64_t spitch, sbs;
    __half* dst;         // element (b, r, c) at dst + b*dbs + r*ldc + c
    int64_t ldc, dbs;
    int64_t rows, cols, batch;
};

// Work items: (row, segment of kCopySeg destination chunks); a destination
// row touches at most (2 cols + 14) / 16 + 1 chunks.
__host__ __device__ inline int64_t unpack_segs(const UnpackArgs& a)
{
    return ((2 * a.cols + 29) / 16 + kCopySeg - 1) / kCopySeg;
}
__host__ __device__ inline int64_t unpack_items(const UnpackArgs& a) { return a.batch * a.rows * unpack_segs(a); }

__global__ void __launch_bounds__(kRepackThreads, kUnpackBlocksPerSm) unpack_rows(const __grid_constant__ UnpackArgs a)
{
    // (as a programmatic dependent of the GEMM: its TMA stores are complete
    // and visible once this returns)
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t segs = unpack_segs(a);
    const int64_t total = unpack_items(a);
    for (int64_t q = warp_index(); q < total; q += warp_count()) {
        const int64_t row = q / segs, seg = q - row * segs;
        const int64_t b = row / a.rows, r = row - b * a.rows;
        copy_row_segment<false>(a.src + b * a.sbs + r * a.spitch, a.dst + b * a.dbs + r * a.ldc, 2 * a.cols,
                                2 * a.cols, seg, lane);
    }
}

}  // namespace gemm_f16_dev
