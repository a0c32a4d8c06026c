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
