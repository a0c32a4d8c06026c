// Host side of the gemm_f16 C ABI: argument checks, the execution plan
// (operand layouts, TMA eligibility, tile width, split-K, grid), tensor-map
// encoding, the split-K workspace and the kernel launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gemm_f16.h"
#include "gemm_kernel.cuh"
#include "repack.cuh"
static_assert(GEMM_F16_MAX_GROUPS == gemm_f16_dev::kMaxGroups, "the header and the kernel agree on the group limit");

using gemm_f16_dev::KernelParams;

// Device status word, written by a kernel that gives up on a bounded wait.
__device__ int g_gemm_f16_status = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxDynSmem = 232448;   // 227 KiB per block on sm_100-class parts
constexpr int kSmemAlignSlack = 1024;

struct DevInfo {
    bool init = false;
    bool supported = false;
    int sms = 0;
    int* status_ptr = nullptr;
    bool smem_attr_set = false;
    int pair_smem = -1;       // cached max_clusters() result for this smem size
    int pair_clusters = 0;
};

std::mutex g_mutex;
DevInfo g_dev[kMaxDevices];

// Library-owned split-K workspace: the partial sums (contents never need to be
// initialised) and the per-tile arrival counters, which start at zero and are
// returned to zero by the last CTA of every tile.
struct Workspace {
    void* partials = nullptr;
    size_t partial_bytes = 0;
    int* counters = nullptr;
    size_t counter_bytes = 0;
    void* repack = nullptr;   // aligned copies of operands TMA cannot address
    size_t repack_bytes = 0;
};
Workspace g_ws[kMaxDevices];

std::atomic<int64_t> g_opt[21];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuMemGetAddressRange_v3020 g_addr_range = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
std::once_flag g_entry_once;

void load_entry_points()
{
    std::call_once(g_entry_once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 3020, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_addr_range = reinterpret_cast<PFN_cuMemGetAddressRange_v3020>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        cudaGetLastError();
    });
}

int64_t opt(int o) { return g_opt[o].load(std::memory_order_relaxed); }

gemm_f16_status device_info(DevInfo** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_F16_ERR_UNSUPPORTED_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_F16_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mutex);
    DevInfo& d = g_dev[dev];
    if (!d.init) {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        d.supported = (major == 10 && minor == 3);
        d.sms = sms;
        void* p = nullptr;
        if (d.supported && cudaGetSymbolAddress(&p, g_gemm_f16_status) == cudaSuccess)
            d.status_ptr = static_cast<int*>(p);
        cudaGetLastError();
        d.init = true;
    }
    *out = &d;
    return d.supported ? GEMM_F16_OK : GEMM_F16_ERR_UNSUPPORTED_DEVICE;
}

// Span of a strided 2-D view in elements: 1 + (r-1)*s_r + (c-1)*s_c.
bool view_extent(int64_t rows, int64_t cols, int64_t s_r, int64_t s_c, int64_t* elems)
{
    int64_t a, b, t;
    if (__builtin_mul_overflow(rows - 1, s_r, &a)) return false;
    if (__builtin_mul_overflow(cols - 1, s_c, &b)) return false;
    if (__builtin_add_overflow(a, b, &t)) return false;
    if (__builtin_add_overflow(t, int64_t(1), &t)) return false;
    if (t > (INT64_MAX / 2)) return false;
    *elems = t;
    return true;
}

bool overlaps(uintptr_t a, int64_t a_bytes, uintptr_t b, int64_t b_bytes)
{
    return a < b + static_cast<uintptr_t>(b_bytes) && b < a + static_cast<uintptr_t>(a_bytes);
}

// The pointer must be device or managed memory of the current device (a peer
// GPU's memory or host memory, pinned or not, is refused), and [p, p+bytes)
// must lie inside the allocation it points into.
bool device_range_ok(const void* p, int64_t bytes)
{
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return false;
    if (at.device != cur) return false;
    if (g_addr_range) {
        CUdeviceptr base = 0;
        size_t size = 0;
        if (g_addr_range(&base, &size, reinterpret_cast<CUdeviceptr>(p)) == CUDA_SUCCESS) {
            const uintptr_t end = static_cast<uintptr_t>(base) + size;
            const uintptr_t q = reinterpret_cast<uintptr_t>(p);
            if (q + static_cast<uintptr_t>(bytes) > end) return false;
        }
    }
    return true;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

struct Args {
    const void* A;
    int64_t sam, sak;
    const void* B;
    int64_t sbk, sbn;
    void* C;
    int64_t ldc, M, N, K;
    // Batched (batch > 1, no group table): problem b at element offsets
    // b*sab, b*sbb, b*scb.  Grouped (rows != nullptr): `batch` groups, group g
    // owning rows rows[g] of the concatenated A and C (M is their sum) and
    // problem g of B at offset g*sbb.
    int64_t batch = 1;
    int64_t sab = 0, sbb = 0, scb = 0;
    const int64_t* rows = nullptr;
    // Fused output stage (`fused`): C = act(A*B + bias), or with Bu (the up
    // projection, read with B's strides and batch stride) the gate/up form
    // act(A*B + bias) * (A*Bu + bias_up).  Bias vectors are fp16, N long,
    // problem (group) b's at element offset b*sbias.
    bool fused = false;
    const void* Bu = nullptr;
    const void* bias = nullptr;
    const void* bias_up = nullptr;
    int64_t sbias = 0;
    int act = 0;
    // The plan may copy an operand TMA cannot address into an aligned buffer
    // of the library workspace (the entry points that own no caller workspace
    // and may allocate).
    bool repack = false;
};

// Elements spanned by `n` copies of a view of `e` elements placed `stride`
// apart (false on overflow).
bool batch_extent(int64_t e, int64_t n, int64_t stride, int64_t* total)
{
    int64_t t;
    if (__builtin_mul_overflow(n - 1, stride, &t) || __builtin_add_overflow(t, e, &t) || t > INT64_MAX / 2) return false;
    *total = t;
    return true;
}

gemm_f16_status validate(const Args& a, bool check_memory, DevInfo** dev)
{
    if (!a.A || !a.B || !a.C) return GEMM_F16_ERR_INVALID_VALUE;
    if (a.M <= 0 || a.N <= 0 || a.K <= 0) return GEMM_F16_ERR_INVALID_VALUE;
    // TMA copy coordinates and the kernel's K-loop coordinates are 32-bit, so
    // each dimension (a grouped call's total rows included) stays below 2^31
    // with room for one tile past the end; element offsets stay 64-bit.
    if (a.M > GEMM_F16_MAX_DIM || a.N > GEMM_F16_MAX_DIM || a.K > GEMM_F16_MAX_DIM) return GEMM_F16_ERR_INVALID_VALUE;
    if (a.sam <= 0 || a.sak <= 0 || a.sbk <= 0 || a.sbn <= 0 || a.ldc < a.N) return GEMM_F16_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B) | reinterpret_cast<uintptr_t>(a.C)) & 1u)
        return GEMM_F16_ERR_INVALID_VALUE;
    if (a.batch < 1 || a.sab < 0 || a.sbb < 0 || a.scb < 0) return GEMM_F16_ERR_INVALID_VALUE;
    if (a.rows && a.batch > gemm_f16_dev::kMaxGroups) return GEMM_F16_ERR_INVALID_VALUE;
    int64_t ea, eb, ec;
    if (!view_extent(a.M, a.K, a.sam, a.sak, &ea) || !view_extent(a.K, a.N, a.sbk, a.sbn, &eb) ||
        !view_extent(a.M, a.N, a.ldc, 1, &ec))
        return GEMM_F16_ERR_INVALID_VALUE;
    if (a.batch > 1) {
        // B (and, batched, A and C) repeat per problem.  The problems' outputs must
        // not overlap: a C stride below one view's span is refused.
        if (!batch_extent(eb, a.batch, a.sbb, &eb)) return GEMM_F16_ERR_INVALID_VALUE;
        if (!a.rows) {
            if (a.scb < ec) return GEMM_F16_ERR_INVALID_VALUE;
            if (!batch_extent(ea, a.batch, a.sab, &ea) || !batch_extent(ec, a.batch, a.scb, &ec))
                return GEMM_F16_ERR_INVALID_VALUE;
        }
    }
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a.A), pb = reinterpret_cast<uintptr_t>(a.B),
                    pc = reinterpret_cast<uintptr_t>(a.C);
    if (overlaps(pc, 2 * ec, pa, 2 * ea) || overlaps(pc, 2 * ec, pb, 2 * eb)) return GEMM_F16_ERR_ALIAS;
    // Fused stage: the up projection spans what B spans; a bias vector N
    // elements per problem.  None of them may overlap C.
    int64_t ebias = a.N;
    if (a.fused) {
        if (a.act < GEMM_F16_ACT_NONE || a.act > GEMM_F16_ACT_GELU || a.sbias < 0) return GEMM_F16_ERR_INVALID_VALUE;
        if (a.bias_up && !a.Bu) return GEMM_F16_ERR_INVALID_VALUE;
        if ((reinterpret_cast<uintptr_t>(a.Bu) | reinterpret_cast<uintptr_t>(a.bias) |
             reinterpret_cast<uintptr_t>(a.bias_up)) & 1u)
            return GEMM_F16_ERR_INVALID_VALUE;
        if (a.batch > 1 && !batch_extent(ebias, a.batch, a.sbias, &ebias)) return GEMM_F16_ERR_INVALID_VALUE;
        if ((a.Bu && overlaps(pc, 2 * ec, reinterpret_cast<uintptr_t>(a.Bu), 2 * eb)) ||
            (a.bias && overlaps(pc, 2 * ec, reinterpret_cast<uintptr_t>(a.bias), 2 * ebias)) ||
            (a.bias_up && overlaps(pc, 2 * ec, reinterpret_cast<uintptr_t>(a.bias_up), 2 * ebias)))
            return GEMM_F16_ERR_ALIAS;
    }
    gemm_f16_status st = device_info(dev);
    if (st != GEMM_F16_OK) return st;
    if (check_memory) {
        load_entry_points();
        if (!device_range_ok(a.A, 2 * ea) || !device_range_ok(a.B, 2 * eb) || !device_range_ok(a.C, 2 * ec))
            return GEMM_F16_ERR_INVALID_VALUE;
        if (a.fused && ((a.Bu && !device_range_ok(a.Bu, 2 * eb)) || (a.bias && !device_range_ok(a.bias, 2 * ebias)) ||
                        (a.bias_up && !device_range_ok(a.bias_up, 2 * ebias))))
            return GEMM_F16_ERR_INVALID_VALUE;
    }
    return GEMM_F16_OK;
}

struct OperandChoice {
    bool tma, mn;
};

// Choose how a kernel-view operand reaches shared memory.  `s_mn`, `s_k` are
// its element strides along the MN and K dimensions, `tile_mn` the tile's MN
// extent.  TMA needs a 16-byte-aligned base, a unit inner stride and an outer
// pitch that is a multiple of 16 bytes.
OperandChoice choose_operand(const void* ptr, int64_t s_mn, int64_t s_k, int64_t MN, int64_t K, int tile_mn,
                             bool allow_tma)
{
    const bool aligned = (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0;
    const int64_t lim = int64_t(1) << 40;
    if (allow_tma && aligned && s_k == 1 && MN < (int64_t(1) << 32) && K < (int64_t(1) << 32)) {
        const int64_t pitch = (MN == 1) ? round_up(2 * K, 16) : 2 * s_mn;
        if (pitch % 16 == 0 && pitch >= 2 * K && pitch < lim) return {true, false};
    }
    if (allow_tma && aligned && s_mn == 1 && tile_mn % 64 == 0 && MN < (int64_t(1) << 32) &&
        K < (int64_t(1) << 32)) {
        const int64_t pitch = (K == 1) ? round_up(2 * MN, 16) : 2 * s_k;
        if (pitch % 16 == 0 && pitch >= 2 * MN && pitch < lim) return {true, true};
    }
    const bool mn = (s_mn == 1 && s_k != 1 && tile_mn % 64 == 0);
    return {false, mn};
}

// `nb` > 0 adds a trailing batch dimension of nb problems `bstride_bytes` apart
// (the box takes one problem).
bool encode_2d(CUtensorMap* tm, const void* ptr, uint64_t inner, uint64_t outer, uint64_t pitch_bytes,
               uint32_t box_inner, uint32_t box_outer, uint64_t nb = 0, uint64_t bstride_bytes = 0)
{
    if (!g_encode) return false;
    cuuint64_t dims[3] = {inner, outer, nb};
    cuuint64_t strides[2] = {pitch_bytes, bstride_bytes};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, nb > 0 ? 3 : 2, const_cast<void*>(ptr), dims, strides,
                          box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// MN-major operand of extent MN (a multiple of 64) as a 3-D tensor: 64
// consecutive MN elements, then K rows `pitch_bytes` apart, then MN / 64
// atom columns 128 bytes apart.  A box of (64, 64, atoms) lands in shared
// memory as `atoms` consecutive 64 x 64 swizzle-atom columns, the layout the
// 2-D form builds with one copy per column.  Every element the map can reach
// lies inside the operand's rows, so no read leaves the MN x K view.
bool encode_3d_mn(CUtensorMap* tm, const void* ptr, uint64_t MN, uint64_t K, uint64_t pitch_bytes, uint32_t atoms,
                  uint64_t nb = 0, uint64_t bstride_bytes = 0)
{
    if (!g_encode || MN % 64 != 0) return false;
    cuuint64_t dims[4] = {64, K, MN / 64, nb};
    cuuint64_t strides[3] = {pitch_bytes, 128, bstride_bytes};
    cuuint32_t box[4] = {64, 64, atoms, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, nb > 0 ? 4 : 3, const_cast<void*>(ptr), dims, strides,
                          box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Operand X' (MN extent mn, K extent K, rows or K rows pitch_bytes apart)
// with the 64-wide K block as an outer dimension, so that one box of two
// blocks lands in two consecutive pipeline slots, each laid out as the
// one-block box would lay it out.  K-major: {64 K, mn, K / 64}, box
// {64, box_mn, 2}; MN-major (mn a multiple of 64): {64 MN, 64 K, mn / 64,
// K / 64}, box {64, 64, box_mn / 64, 2}; then the batch dimension, if any.
// Only whole K blocks are addressable: a ragged last block, whose missing
// columns a box must zero-fill, is read through the one-block map.
bool encode_two_k(CUtensorMap* tm, const void* ptr, bool mn_major, uint64_t mn, uint64_t K, uint64_t pitch_bytes,
                  uint32_t box_mn, uint64_t nb, uint64_t bstride_bytes)
{
    if (!g_encode || K < 128 || (mn_major && mn % 64 != 0)) return false;
    cuuint64_t dims[5] = {64, mn, K / 64, 0, 0};
    cuuint64_t strides[4] = {pitch_bytes, 128, 0, 0};
    cuuint32_t box[5] = {64, box_mn, 2, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    int rank = 3;
    if (mn_major) {
        dims[1] = 64, dims[2] = mn / 64, dims[3] = K / 64;
        strides[2] = 64 * pitch_bytes;
        box[1] = 64, box[2] = box_mn / 64, box[3] = 2;
        rank = 4;
    }
    if (nb > 0) {
        dims[rank] = nb;
        strides[rank - 1] = bstride_bytes;
        ++rank;
    }
    CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr),
                          dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct Plan {
    gemm_f16_plan pub;
    bool fused;   // launch the kernels with the fused output stage
    int ncopies;  // repack copies to run before the GEMM (A', B', up projection)
    gemm_f16_dev::RepackArgs copies[3];
    bool unpack;  // C goes through an aligned buffer, then this copy moves it into place
    gemm_f16_dev::UnpackArgs out;
    KernelParams kp;
    size_t counter_bytes;   // split-K counters: align256(4 * tiles)
    size_t partial_bytes;   // split-K partials: align256(4 * units * tile_m * tile_n)
};

// Blocks of 8 warps for a copy of `items` work items (one item per warp and
// pass): at most the resident blocks of every SM, one wave.
unsigned copy_blocks(int64_t items, int sms, int per_sm)
{
    return static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>((items + 7) / 8, static_cast<int64_t>(sms) * per_sm)));
}

bool set_smem_attributes(DevInfo& dev)
{
    std::lock_guard<std::mutex> lk(g_mutex);
    if (dev.smem_attr_set) return true;
    using namespace gemm_f16_dev;
    const void* kernels[] = {reinterpret_cast<const void*>(gemm_f16_persistent<false, false>),
                             reinterpret_cast<const void*>(gemm_f16_persistent<true, false>),
                             reinterpret_cast<const void*>(gemm_f16_persistent<false, true>),
                             reinterpret_cast<const void*>(gemm_f16_persistent<true, true>),
                             reinterpret_cast<const void*>(gemm_f16_persistent<false, true, true>),
                             reinterpret_cast<const void*>(gemm_f16_persistent<true, true, true>)};
    bool ok = true;
    for (const void* k : kernels)
        ok = ok && cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return false;
    }
    dev.smem_attr_set = true;
    return true;
}

// How many clusters of two CTAs (the pair form) can be resident at once.
// Clusters must fit inside a GPC, so this can be less than half the SM count.
int max_clusters(DevInfo& dev, int smem)
{
    constexpr int size = 2;
    if (!set_smem_attributes(dev)) return 0;
    {
        std::lock_guard<std::mutex> lk(g_mutex);
        if (dev.pair_smem == smem) return dev.pair_clusters;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(size * (dev.sms / size));
    cfg.blockDim = dim3(gemm_f16_dev::kNumThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, gemm_f16_dev::gemm_f16_persistent<true, false>, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    std::lock_guard<std::mutex> lk(g_mutex);
    dev.pair_smem = smem;
    dev.pair_clusters = n;
    return n;
}

// Classic split-K (every tile cut into `splits` equal K segments) runs only
// when forced through GEMM_F16_OPT_SPLITS; otherwise the schedule below uses
// stream-K to fill the device.
int choose_splits(int kblocks)
{
    const int64_t forced = opt(GEMM_F16_OPT_SPLITS);
    return forced > 0 ? static_cast<int>(std::min<int64_t>(forced, kblocks)) : 1;
}

// K segments per tile that a swapped small-M pair plan runs by default (1:
// none).  With fewer tiles T than clusters W (sms / 2) but at least half as
// many, S in {2, 3, 4} segments make S*T units in ceil(S*T / W) waves; the S
// that fills its waves best (ties: the smaller S) is taken when it fills them
// to at least 80 % and leaves each segment 8 K blocks or more; neither
// split-K nor stream-K may be forced.  16 x N x 8192, L2 flushed, us per call
// for the best S against stream-K: 48 tiles 45.9 (S 3) vs 47.2, 56 tiles
// 50.6 (S 4) vs 52.8, 64 tiles 52.8 (S 2) vs 56.2; at 40 tiles the best fill
// is 0.79 (S 3: 43.7) and stream-K (43.0) stays.  The unit order, K segment
// first, is what pays (64 tiles, S 2, tile-major order: 56.3).
int kseg_default(bool swap, bool pair, bool gated, int64_t tiles, int kblocks, int sms)
{
    const int64_t W = sms / 2;
    if (!swap || !pair || gated || opt(GEMM_F16_OPT_SPLITS) != 0 || opt(GEMM_F16_OPT_STREAMK) != 0 || tiles >= W ||
        2 * tiles < W)
        return 1;
    int best = 1;
    double best_fill = 0.8 - 1e-9;
    for (int S = 2; S <= 4; ++S) {
        if (kblocks < 8 * S) break;
        const int64_t units = S * tiles, waves = (units + W - 1) / W;
        const double fill = static_cast<double>(units) / static_cast<double>(waves * W);
        if (fill > best_fill + 1e-9) {
            best_fill = fill;
            best = S;
        }
    }
    return best;
}

// How the tiles are spread over the persistent workers (CTAs, or 2-CTA
// clusters in the pair form).  With W workers and T tiles of KB K blocks:
//  - classic split-K (forced): T*splits equal units, round-robin;
//  - T a multiple of W, or too little work to cut: whole tiles, round-robin;
//  - otherwise data-parallel waves of whole tiles for all but the last
//    1 + (T mod W)/W waves, whose K blocks are spread evenly over all W workers
//    (stream-K; TileLang tutorial ch. 14, section 4.2), so every worker gets
//    the same number of K blocks.  Tiles cut by a worker boundary are summed by
//    the last of their workers to finish, in K order.
struct Schedule {
    int workers = 1, num_units = 0, sk_tile0 = 0, nseg_max = 0, sk_slot_base = 0;
    int64_t sk_iters = 0;
    int64_t partial_slots = 0;   // fp32 tile partials the workspace must hold (per CTA rank)
    int tail_tile0 = INT32_MAX, tail_split = 1;
};

// Tail split: with whole tiles only, the last wave holds T mod W tiles and
// leaves the other workers idle.  Cutting those tiles along N into s pieces
// (each still a complete K reduction of its columns, so no partial sums) makes
// that wave ceil(s*rem/W)/s tile-times long; take the smallest s that helps.
// A piece keeps at least `min_bn` columns and a multiple of 64.
void tail_split(Schedule& s, int64_t tiles, int BN, int min_bn, int64_t W)
{
    if (opt(GEMM_F16_OPT_TAIL_SPLIT) == 1) return;
    const int64_t rem = tiles % W;
    if (rem == 0) return;
    int best = 1;
    double best_t = 1.0;
    for (int sp = 2; BN % sp == 0 && BN / sp >= min_bn && (BN / sp) % 64 == 0; sp *= 2) {
        const double t = static_cast<double>((rem * sp + W - 1) / W) / sp;
        if (t < best_t - 1e-9) {
            best_t = t;
            best = sp;
        }
    }
    if (best == 1) return;
    s.tail_tile0 = static_cast<int>(tiles - rem);
    s.tail_split = best;
    s.num_units = static_cast<int>(tiles - rem + rem * best);
    s.workers = static_cast<int>(std::min<int64_t>(s.num_units, W));
}

Schedule make_schedule(int64_t tiles, int kblocks, int splits, int max_workers, int BN, int min_bn, bool streamk)
{
    Schedule s;
    if (splits > 1) {
        s.num_units = static_cast<int>(tiles * splits);
        s.workers = static_cast<int>(std::min<int64_t>(s.num_units, max_workers));
        s.partial_slots = s.num_units;
        return s;
    }
    s.num_units = static_cast<int>(tiles);
    s.workers = static_cast<int>(std::min<int64_t>(tiles, max_workers));
    const int64_t W = max_workers;
    if (!streamk) {
        tail_split(s, tiles, BN, min_bn, W);
        return s;
    }
    if (tiles % W == 0) return s;
    const int64_t full = tiles / W;
    const int64_t sk_tiles = full >= 1 ? tiles % W + W : tiles;
    const int64_t S = sk_tiles * kblocks;
    // When the tiles alone cannot fill the device: at least 8 K blocks per
    // worker, at most 16 workers per tile (the last one adds their partials),
    // and more workers than tiles.
    const int64_t w = full >= 1 ? W : std::min<int64_t>(std::min<int64_t>(W, S / 8), sk_tiles * 16);
    if (w <= sk_tiles && full == 0) return s;
    if (S < 4 * w) return s;
    s.workers = static_cast<int>(w);
    s.num_units = static_cast<int>(tiles - sk_tiles);
    s.sk_tile0 = s.num_units;
    s.sk_iters = S;
    // Partial slots are numbered per tile: stream-K tile t keeps its units'
    // partials in slots t*nseg_max .. t*nseg_max + (units covering t) - 1.
    auto worker_of = [&](int64_t x) {   // the worker whose range holds stream-K block x
        return std::min<int64_t>(((x + 1) * w + S - 1) / S - 1, w - 1);
    };
    int64_t most = 1;
    for (int64_t t = 0; t < sk_tiles; ++t)
        most = std::max<int64_t>(most, worker_of(t * kblocks + kblocks - 1) - worker_of(t * kblocks) + 1);
    s.nseg_max = static_cast<int>(most);
    s.sk_slot_base = 0;
    s.partial_slots = sk_tiles * most;
    return s;
}

void shape_plan(int64_t M, int64_t N, int64_t K, int sms, bool allow_swap, bool* swap, int64_t* Mv, int64_t* Nv,
                int* BN, int* tiles_m, int* tiles_n, int* kblocks, int* splits)
{
    const int64_t sw = opt(GEMM_F16_OPT_SWAP);
    *swap = allow_swap && ((sw == 2) || (sw == 0 && M <= 64 && N >= 2 * M));
    *Mv = *swap ? N : M;
    *Nv = *swap ? M : N;
    int bn;
    if (*swap) {
        bn = static_cast<int>(round_up(*Nv, 16));
        if (bn > 256) bn = 256;
    } else {
        const int64_t forced = opt(GEMM_F16_OPT_TILE_N);
        bn = forced > 0 ? static_cast<int>(forced) : static_cast<int>(std::min<int64_t>(256, round_up(*Nv, 64)));
    }
    *BN = bn;
    *tiles_m = static_cast<int>((*Mv + gemm_f16_dev::kBM - 1) / gemm_f16_dev::kBM);
    *tiles_n = static_cast<int>((*Nv + bn - 1) / bn);
    *kblocks = static_cast<int>((K + gemm_f16_dev::kBK - 1) / gemm_f16_dev::kBK);
    (void)sms;
    *splits = choose_splits(*kblocks);
}

// Caller-workspace layout: [counters, align256(4*tiles*ranks)] [partials].
// `ranks` is 2 for the pair form (each CTA of a pair keeps its own 128 rows).
size_t workspace_bytes_for(int64_t slots, int BN, int64_t tiles, int ranks, size_t* counter_bytes,
                           size_t* partial_bytes)
{
    const size_t cb = static_cast<size_t>(round_up(tiles * ranks * 4, 256));
    const size_t pb = static_cast<size_t>(round_up(slots * ranks * gemm_f16_dev::kBM * BN * 4, 256));
    if (counter_bytes) *counter_bytes = cb;
    if (partial_bytes) *partial_bytes = pb;
    return cb + pb;
}

// Device buffer of `bytes` for repacked operands: the library workspace's, or
// (plan_only) a stand-in aligned address that is never dereferenced.
void* repack_buffer(size_t bytes, bool plan_only, cudaStream_t stream);

// Products below this many FLOPs gather unaligned operands in the kernel: the
// copy's extra launch and traffic would not pay for itself.
constexpr double kRepackMinFlops = 1e9;

gemm_f16_status make_plan(const Args& a, const DevInfo& dev, Plan* pl, bool plan_only = false,
                          cudaStream_t stream = nullptr)
{
    std::memset(pl, 0, sizeof(*pl));
    KernelParams& kp = pl->kp;
    gemm_f16_plan& pub = pl->pub;
    bool swap;
    int64_t Mv, Nv;
    int BN, tiles_m, tiles_n, kblocks, splits;
    const bool grouped = a.rows != nullptr;
    const bool batched = !grouped && a.batch > 1;
    const bool gated = a.fused && a.Bu != nullptr;
    // (groups differ in M, so the swapped form, which tiles over M as N, is not
    // used; nor for the gate/up form, whose two products share the MMA's N)
    shape_plan(a.M, a.N, a.K, dev.sms, !grouped && !gated, &swap, &Mv, &Nv, &BN, &tiles_m, &tiles_n, &kblocks,
               &splits);
    // Gate/up: tiles of `out` output columns whose accumulator holds 2*out
    // columns (gate then up); whole tiles only.
    int out_cols = BN;
    if (gated) {
        const int64_t forced = opt(GEMM_F16_OPT_TILE_N);
        out_cols = forced > 0 ? static_cast<int>(std::min<int64_t>(forced, 128))
                              : static_cast<int>(std::min<int64_t>(128, round_up(a.N, 64)));
        BN = 2 * out_cols;
        tiles_n = static_cast<int>((a.N + out_cols - 1) / out_cols);
        splits = 1;
    }
    if (BN < 16 || BN > 256 || BN % 16 != 0) return GEMM_F16_ERR_INVALID_VALUE;

    // Kernel view: C'[m,n] = sum_k A'[m,k] B'[k,n].
    if (!swap) {
        kp.A = static_cast<const __half*>(a.A), kp.a_sm = a.sam, kp.a_sk = a.sak;
        kp.B = static_cast<const __half*>(a.B), kp.b_sk = a.sbk, kp.b_sn = a.sbn;
        kp.C = static_cast<__half*>(a.C), kp.c_sm = a.ldc, kp.c_sn = 1;
    } else {   // C^T = B^T A^T
        kp.A = static_cast<const __half*>(a.B), kp.a_sm = a.sbn, kp.a_sk = a.sbk;
        kp.B = static_cast<const __half*>(a.A), kp.b_sk = a.sak, kp.b_sn = a.sam;
        kp.C = static_cast<__half*>(a.C), kp.c_sm = 1, kp.c_sn = a.ldc;
    }
    kp.M = Mv, kp.N = Nv, kp.K = a.K;
    // Batch strides of the kernel view; an operand shared by every problem
    // (stride 0) needs no batch dimension.
    int64_t a_bs = 0, b_bs = 0, c_bs = 0;
    if (batched) {
        a_bs = swap ? a.sbb : a.sab;
        b_bs = swap ? a.sab : a.sbb;
        c_bs = a.scb;
    } else if (grouped) {
        b_bs = a.sbb;
    }
    const bool a_bd = batched && a_bs > 0;
    const bool b_bd = (batched || grouped) && a.batch > 1 && b_bs > 0;
    const bool c_bd = batched;
    auto bs_ok = [](int64_t bs) { return (2 * bs) % 16 == 0 && 2 * bs < (int64_t(1) << 40); };   // TMA stride rules

    const int64_t fg = opt(GEMM_F16_OPT_FORCE_GATHER);
    load_entry_points();
    const bool have_tma = g_encode != nullptr;
    OperandChoice ca = choose_operand(kp.A, kp.a_sm, kp.a_sk, Mv, a.K, gemm_f16_dev::kBM,
                                      have_tma && !(fg & 1) && (!a_bd || bs_ok(a_bs)));
    // Grouped: an MN-major A box starts at its group's first row (+ a multiple
    // of 128), and that row is the box's innermost (x) coordinate, which TMA
    // needs on a 16-byte boundary.  Unless every non-empty group starts on a
    // multiple of 8 rows, A is not read MN-major through TMA (it is gathered, or
    // copied K-major below).
    bool a_mn_tma_ok = true;
    // (the one-copy 3-D box of an MN-major A addresses whole 64-row swizzle
    // atoms, so a grouped A takes it only when every group starts on one)
    bool a_3d_groups_ok = true;
    if (grouped) {
        int64_t r0 = 0;
        for (int64_t g = 0; g < a.batch; ++g) {
            if (a.rows[g] > 0 && r0 % 8 != 0) a_mn_tma_ok = false;
            if (a.rows[g] > 0 && r0 % 64 != 0) a_3d_groups_ok = false;
            r0 += a.rows[g];
        }
    }
    if (ca.tma && ca.mn && !a_mn_tma_ok)
        ca = choose_operand(kp.A, kp.a_sm, kp.a_sk, Mv, a.K, gemm_f16_dev::kBM, false);
    OperandChoice cb = choose_operand(kp.B, kp.b_sn, kp.b_sk, Nv, a.K, gated ? out_cols : BN,
                                      have_tma && !(fg & 2) && (!b_bd || bs_ok(b_bs)));
    if (gated) {
        // both projections take the same path (same strides; only the bases differ)
        kp.Bu = static_cast<const __half*>(a.Bu);
        const OperandChoice cu = choose_operand(kp.Bu, kp.b_sn, kp.b_sk, Nv, a.K, out_cols,
                                                have_tma && !(fg & 2) && (!b_bd || bs_ok(b_bs)));
        if (cu.tma != cb.tma || cu.mn != cb.mn) cb = choose_operand(kp.B, kp.b_sn, kp.b_sk, Nv, a.K, out_cols, false);
    }

    // Padding form of the boundary handling (AI-infra page, section 05): an
    // operand TMA cannot address (unaligned base or pitch, no unit stride) is
    // copied once into an aligned buffer whose rows run along its smaller
    // stride, when the product is large enough; the gather stays for small
    // products, forced gathers and the entry points that may not allocate.
    pl->ncopies = 0;
    int repacked = 0;
    // MN extent the 3-D box maps see: the operand's, or for an MN-major copy
    // its rows rounded up to whole 64-element atoms (the copy's pitch covers
    // them and the copy zero-fills them), so that the copy always takes the
    // one-box-per-stage form.
    int64_t a_mn_ext = Mv, b_mn_ext = Nv;
    {
        const int64_t rp = opt(GEMM_F16_OPT_REPACK);
        const double work = 2.0 * static_cast<double>(Mv) * static_cast<double>(Nv) * static_cast<double>(a.K) *
                            static_cast<double>(batched ? a.batch : 1);
        const bool want_a = !ca.tma && !(fg & 1), want_b = !cb.tma && !(fg & 2);
        // C that TMA cannot store in place (unaligned base or pitch, or N not a
        // multiple of 8) but whose tiles could go out by TMA: stored into an
        // aligned buffer and moved into place by the unpack copy.
        const bool c_in_place = a.N % 8 == 0 && (reinterpret_cast<uintptr_t>(a.C) & 15u) == 0 &&
                                (a.ldc * 2) % 16 == 0 && (a.ldc * 2) < (int64_t(1) << 40) && (!c_bd || bs_ok(c_bs));
        const bool want_c = !c_in_place && !(fg & 4) && !swap && splits == 1 && out_cols % 64 == 0 &&
                            a.M < (int64_t(1) << 32) && a.N < (int64_t(1) << 32);
        if (a.repack && have_tma && rp != 1 && (rp == 2 || work >= kRepackMinFlops) && (want_a || want_b || want_c)) {
            struct Layout {
                bool mn;   // rows of the copy run along MN (MN-major result)
                int64_t rows, cols, s_r, s_c, pitch, nb, s_b;
            };
            auto layout = [&](int64_t s_mn, int64_t s_k, int64_t MN, int64_t bs, bool bd) {
                Layout l;
                l.mn = s_mn == 1 || (s_k != 1 && s_mn <= s_k);
                l.rows = l.mn ? a.K : MN;
                l.cols = l.mn ? MN : a.K;
                l.s_r = l.mn ? s_k : s_mn;
                l.s_c = l.mn ? s_mn : s_k;
                // (MN-major copies: whole 64-element swizzle atoms per row)
                l.pitch = round_up(l.cols, l.mn ? 64 : 8);
                l.nb = bd ? a.batch : 1;
                l.s_b = bd ? bs : 0;
                return l;
            };
            Layout la = layout(kp.a_sm, kp.a_sk, Mv, a_bs, a_bd);
            if (la.mn && !a_mn_tma_ok) {   // copy A K-major: rows of K along the rows of C
                la.mn = false;
                la.rows = Mv, la.cols = a.K, la.s_r = kp.a_sm, la.s_c = kp.a_sk;
                la.pitch = round_up(a.K, 8);
            }
            const Layout lb = layout(kp.b_sn, kp.b_sk, Nv, b_bs, b_bd);
            const int tile_b = gated ? out_cols : BN;
            // the copy must be TMA-addressable (an MN-major copy needs 64-wide tiles)
            const bool do_a = want_a && (!la.mn || gemm_f16_dev::kBM % 64 == 0);
            const bool do_b = want_b && (!lb.mn || tile_b % 64 == 0);
            auto bytes_of = [](const Layout& l) {
                return static_cast<size_t>(round_up(2 * l.nb * l.rows * l.pitch, 256));
            };
            // the aligned C buffer: rows of C, pitch N rounded up to 8 elements
            const int64_t c_pitch = round_up(a.N, 8), c_nb = c_bd ? a.batch : 1;
            const size_t c_bytes = want_c ? static_cast<size_t>(round_up(2 * c_nb * a.M * c_pitch, 256)) : 0;
            const size_t need =
                (do_a ? bytes_of(la) : 0) + (do_b ? (gated ? 2 : 1) * bytes_of(lb) : 0) + c_bytes;
            char* buf = need ? static_cast<char*>(repack_buffer(need, plan_only, stream)) : nullptr;
            if (need && !buf) return GEMM_F16_ERR_OUT_OF_MEMORY;
            auto add_copy = [&](const Layout& l, const __half* src) {
                gemm_f16_dev::RepackArgs& c = pl->copies[pl->ncopies++];
                c.src = src, c.s_r = l.s_r, c.s_c = l.s_c, c.s_b = l.s_b;
                c.dst = reinterpret_cast<__half*>(buf);
                c.pitch = l.pitch, c.dst_bs = l.rows * l.pitch;
                c.rows = l.rows, c.cols = l.cols, c.batch = l.nb;
                buf += bytes_of(l);
                return c.dst;
            };
            if (do_a) {
                kp.A = add_copy(la, kp.A);
                kp.a_sm = la.mn ? 1 : la.pitch;
                kp.a_sk = la.mn ? la.pitch : 1;
                if (a_bd) a_bs = la.rows * la.pitch;
                ca = choose_operand(kp.A, kp.a_sm, kp.a_sk, Mv, a.K, gemm_f16_dev::kBM,
                                    have_tma && (!a_bd || bs_ok(a_bs)));
                if (la.mn) a_mn_ext = round_up(Mv, 64);
                repacked |= 1;
            }
            if (do_b) {
                kp.B = add_copy(lb, kp.B);
                if (gated) kp.Bu = add_copy(lb, kp.Bu);
                kp.b_sn = lb.mn ? 1 : lb.pitch;
                kp.b_sk = lb.mn ? lb.pitch : 1;
                if (b_bd) b_bs = lb.rows * lb.pitch;
                cb = choose_operand(kp.B, kp.b_sn, kp.b_sk, Nv, a.K, tile_b, have_tma && (!b_bd || bs_ok(b_bs)));
                if (lb.mn) b_mn_ext = round_up(Nv, 64);
                repacked |= 2;
            }
            if (want_c) {
                // the kernel writes C' into the aligned buffer (by TMA, and the
                // few per-thread stores a grouped tile may take); the unpack copy
                // then writes only the M x N view of the caller's C
                __half* cs = reinterpret_cast<__half*>(buf);
                gemm_f16_dev::UnpackArgs& u = pl->out;
                u.src = cs, u.spitch = c_pitch, u.sbs = a.M * c_pitch;
                u.dst = static_cast<__half*>(a.C), u.ldc = a.ldc, u.dbs = c_bd ? a.scb : 0;
                u.rows = a.M, u.cols = a.N, u.batch = c_nb;
                pl->unpack = true;
                kp.C = cs, kp.c_sm = c_pitch, kp.c_sn = 1;
                if (c_bd) c_bs = a.M * c_pitch;
                repacked |= 4;
            }
        }
    }

    // Pair form (two CTAs per 256 x BN tile): TMA operands, no split-K, and a
    // B half that is a whole number of 64-column swizzle atoms.
    const int64_t pair_opt = opt(GEMM_F16_OPT_PAIR);
    // The swapped small-M form pairs too when its B' (the caller's A) is
    // K-major: M = 256 per MMA, each CTA loading BN / 2 (>= 8) rows of B'; the
    // two CTAs of a pair then read adjacent 256-byte pieces of each row of the
    // streamed operand together.  16 x 16384 x 8192: 56.8 instead of 57.3 us
    // per call with L2 flushed.
    const bool swap_pair = swap && pair_opt != 1 && !cb.mn && BN % 16 == 0;
    const bool pair = pair_opt != 1 && (!swap || swap_pair) && (splits == 1 || pair_opt == 2) && ca.tma && cb.tma &&
                      (BN == 256 || (pair_opt == 2 && BN == 128) || swap_pair) && Mv > gemm_f16_dev::kBM;
    const int tile_rows = pair ? 2 * gemm_f16_dev::kBM : gemm_f16_dev::kBM;
    const int bcols = pair ? BN / 2 : BN;   // B columns one CTA loads
    if (pair) tiles_m = static_cast<int>((Mv + tile_rows - 1) / tile_rows);
    int64_t tiles = static_cast<int64_t>(tiles_m) * tiles_n * (batched ? a.batch : 1);
    if (grouped) {   // per group: ceil(rows / tile_rows) tile rows; tiles numbered group by group
        int64_t t0 = 0, row0 = 0;
        for (int64_t g = 0; g < a.batch; ++g) {
            const int64_t tm = (a.rows[g] + tile_rows - 1) / tile_rows;
            if (t0 > INT32_MAX / 4) return GEMM_F16_ERR_INVALID_VALUE;
            kp.g_tile0[g] = static_cast<int>(t0);
            kp.g_tm[g] = static_cast<int>(tm);
            kp.g_row0[g] = row0;
            kp.g_rows[g] = a.rows[g];
            t0 += tm * tiles_n;
            row0 += a.rows[g];
        }
        kp.g_tile0[a.batch] = static_cast<int>(t0);
        tiles = t0;
    }
    if (tiles * splits > INT32_MAX / 4 || tiles * kblocks > (int64_t(1) << 40)) return GEMM_F16_ERR_INVALID_VALUE;
    kp.gmode = grouped ? 2 : (batched ? 1 : 0);
    kp.groups = static_cast<int>(a.batch);
    kp.a_bs = a_bs, kp.b_bs = b_bs, kp.c_bs = c_bs;

    bool a_3d = false, b_3d = false;
    // trailing batch dimensions (0: none)
    const uint64_t nb_a = a_bd ? a.batch : 0, bst_a = a_bd ? 2 * a_bs : 0;
    const uint64_t nb_b = b_bd ? a.batch : 0, bst_b = b_bd ? 2 * b_bs : 0;
    if (ca.tma) {
        a_3d = ca.mn && (!grouped || a_3d_groups_ok) &&
               encode_3d_mn(&kp.tmA, kp.A, a_mn_ext, a.K, a.K == 1 ? round_up(2 * Mv, 16) : 2 * kp.a_sk,
                                     gemm_f16_dev::kBM / 64, nb_a, bst_a);
        const bool ok = a_3d ? true
                        : ca.mn ? encode_2d(&kp.tmA, kp.A, Mv, a.K, a.K == 1 ? round_up(2 * Mv, 16) : 2 * kp.a_sk, 64, 64,
                                            nb_a, bst_a)
                              : encode_2d(&kp.tmA, kp.A, a.K, Mv, Mv == 1 ? round_up(2 * a.K, 16) : 2 * kp.a_sm, 64,
                                          gemm_f16_dev::kBM, nb_a, bst_a);
        if (!ok) {
            if (pair) return GEMM_F16_ERR_LAUNCH;
            ca = choose_operand(kp.A, kp.a_sm, kp.a_sk, Mv, a.K, gemm_f16_dev::kBM, false);
        }
    }
    // B's box: a CTA's whole share of the tile's columns.  The gate/up form
    // reads boxes of its output width from both projections.
    auto encode_b = [&]() {
        const int cols = gated ? out_cols : bcols;
        auto enc = [&](CUtensorMap* tm, const __half* ptr) {
            b_3d = cb.mn && encode_3d_mn(tm, ptr, b_mn_ext, a.K, a.K == 1 ? round_up(2 * Nv, 16) : 2 * kp.b_sk,
                                         static_cast<uint32_t>(cols / 64), nb_b, bst_b);
            return b_3d ? true
                   : cb.mn ? encode_2d(tm, ptr, Nv, a.K, a.K == 1 ? round_up(2 * Nv, 16) : 2 * kp.b_sk, 64, 64, nb_b,
                                       bst_b)
                           : encode_2d(tm, ptr, a.K, Nv, Nv == 1 ? round_up(2 * a.K, 16) : 2 * kp.b_sn, 64,
                                       static_cast<uint32_t>(cols), nb_b, bst_b);
        };
        return enc(&kp.tmB, kp.B) && (!gated || enc(&kp.tmBu, kp.Bu));
    };
    if (cb.tma) {
        if (!encode_b()) {
            if (pair) return GEMM_F16_ERR_LAUNCH;
            cb = choose_operand(kp.B, kp.b_sn, kp.b_sk, Nv, a.K, gated ? out_cols : BN, false);
        }
    }
    // TMA stores write whole 16-byte chunks at the N edge, so a C row whose
    // width is not a multiple of 8 elements would get its pitch padding
    // overwritten: such a C goes through the masked stores.
    bool c_tma = pl->unpack ||
                 (have_tma && !(fg & 4) && !swap && splits == 1 && out_cols % 64 == 0 && a.N % 8 == 0 &&
                  (reinterpret_cast<uintptr_t>(a.C) & 15u) == 0 && (a.ldc * 2) % 16 == 0 && a.M < (int64_t(1) << 32) &&
                  a.N < (int64_t(1) << 32) && (a.ldc * 2) < (int64_t(1) << 40) && (!c_bd || bs_ok(c_bs)));
    if (c_tma)   // (kp.C / kp.c_sm: the caller's C, or the aligned buffer); boxes of one warp's and of the CTA's rows
        c_tma = encode_2d(&kp.tmC, kp.C, a.N, a.M, 2 * kp.c_sm, 64, 32, c_bd ? a.batch : 0, c_bd ? 2 * c_bs : 0) &&
                encode_2d(&kp.tmC4, kp.C, a.N, a.M, 2 * kp.c_sm, 64, 128, c_bd ? a.batch : 0, c_bd ? 2 * c_bs : 0);
    if (pl->unpack && !c_tma) return GEMM_F16_ERR_LAUNCH;
    kp.a_bdim = (ca.tma && a_bd) ? 1u : 0u;
    kp.b_bdim = (cb.tma && b_bd) ? 1u : 0u;
    kp.c_bdim = (c_tma && c_bd) ? 1u : 0u;
    // Two K blocks per copy: both operands by TMA in a layout the one-block
    // maps read with a single box per slot (K-major, or MN-major as 3-D boxes).
    kp.k2 = 0;
    kp.kfull = static_cast<int>(a.K / 64);
    // (The single-CTA gate/up stage interleaves gate and up boxes per slot, a
    // layout one two-block box cannot write; its pair form splits them over
    // the two CTAs.)
    if (opt(GEMM_F16_OPT_TWO_K_LOADS) != 1 && (!gated || pair) && ca.tma && cb.tma && (!ca.mn || a_3d) &&
        (!cb.mn || b_3d) && a.K >= 128) {
        const uint64_t pitch_b = cb.mn ? 2 * kp.b_sk : (Nv == 1 ? round_up(2 * a.K, 16) : 2 * kp.b_sn);
        const uint32_t box_b = static_cast<uint32_t>(gated ? out_cols : bcols);
        const bool ok =
            encode_two_k(&kp.tmA2k, kp.A, ca.mn, ca.mn ? a_mn_ext : Mv, a.K,
                         ca.mn ? 2 * kp.a_sk : (Mv == 1 ? round_up(2 * a.K, 16) : 2 * kp.a_sm), gemm_f16_dev::kBM, nb_a,
                         bst_a) &&
            encode_two_k(&kp.tmB2k, kp.B, cb.mn, cb.mn ? b_mn_ext : Nv, a.K, pitch_b, box_b, nb_b, bst_b) &&
            (!gated || encode_two_k(&kp.tmBu2k, kp.Bu, cb.mn, cb.mn ? b_mn_ext : Nv, a.K, pitch_b, box_b, nb_b, bst_b));
        kp.k2 = ok ? 1u : 0u;
    }

    const uint32_t stage_b = static_cast<uint32_t>(bcols) * gemm_f16_dev::kBK * 2;
    const uint32_t stage_bytes = gemm_f16_dev::kStageABytes + stage_b;
    // The 32 KB epilogue buffer stages TMA stores of C, and is where the last
    // unit of a tile cut along K collects the other units' partials.
    // K segments for a swapped small-M pair plan whose tiles are fewer than the
    // clusters but at least half as many (kseg_default): every cluster then
    // streams a segment of the large operand, and the segment-major unit order
    // has the clusters read the same rows of it at the same time.
    if (splits == 1) splits = kseg_default(swap, pair, gated, tiles, kblocks, dev.sms);
    // Stream-K: forced by GEMM_F16_OPT_STREAMK = 2, and the default when an
    // operand is gathered (gathered tiles are slow, so balancing the last wave
    // pays for the fixup) and for other swapped small-M plans with fewer tiles
    // than SMs (the product streams the large operand from HBM, and stream-K
    // lets every SM stream a share); otherwise the last partial wave is split
    // along N.
    const int64_t sk_opt = opt(GEMM_F16_OPT_STREAMK);
    const bool sk_default = !ca.tma || !cb.tma || (swap && tiles < dev.sms);
    const bool use_sk = splits == 1 && !gated && (sk_opt == 2 || (sk_opt == 0 && sk_default));
    const bool may_cut = splits > 1 || use_sk;
    // A C that TMA cannot store but whose columns are contiguous is staged in
    // the same buffer and written row by row by the epilogue warps.
    const bool c_stage = !c_tma && !swap;
    const int epi = (c_tma || c_stage || may_cut) ? static_cast<int>(gemm_f16_dev::kEpiBytes) : 0;
    int stages = (kMaxDynSmem - kSmemAlignSlack - epi - static_cast<int>(gemm_f16_dev::kBarrierBytes)) /
                 static_cast<int>(stage_bytes);
    stages = std::min(stages, gemm_f16_dev::kMaxStages);
    if (opt(GEMM_F16_OPT_MAX_STAGES) >= 2) stages = std::min<int>(stages, static_cast<int>(opt(GEMM_F16_OPT_MAX_STAGES)));
    stages -= stages % gemm_f16_dev::kSlots;   // whole barrier phases of kSlots slots
    if (stages < gemm_f16_dev::kSlots) return GEMM_F16_ERR_INVALID_VALUE;
    const int smem = kSmemAlignSlack + stages * static_cast<int>(stage_bytes) + epi +
                     static_cast<int>(gemm_f16_dev::kBarrierBytes);

    // Persistent workers: CTAs, or clusters of 2 CTAs in the pair form.
    const int64_t cap = opt(GEMM_F16_OPT_MAX_CTAS);
    int64_t max_workers = dev.sms;
    const int cluster_ctas = pair ? 2 : 1;
    if (pair) max_workers = max_clusters(const_cast<DevInfo&>(dev), smem);
    if (cap > 0) max_workers = std::min<int64_t>(max_workers, std::max<int64_t>(1, cap / cluster_ctas));
    if (max_workers < 1) return GEMM_F16_ERR_LAUNCH;
    // Narrowest tail piece: the pair form keeps >= 64 B columns per CTA; a
    // TMA-stored C needs whole 64-column boxes.  (gate/up tiles are never cut:
    // the minimum piece is wider than the tile)
    const Schedule sch = make_schedule(tiles, kblocks, splits, static_cast<int>(max_workers), BN,
                                       gated ? 2 * BN : (pair ? 128 : 64), use_sk);
    const int grid = cluster_ctas * sch.workers;
    const int64_t panel = opt(GEMM_F16_OPT_PANEL);

    kp.status = dev.status_ptr;
    const int64_t tmo = opt(GEMM_F16_OPT_TIMEOUT_MS);
    kp.timeout_ns = static_cast<uint64_t>(tmo > 0 ? tmo : 1000) * 1000000ull;
    kp.tiles_m = tiles_m, kp.tiles_n = tiles_n, kp.splits = splits, kp.kblocks = kblocks;
    kp.num_units = sch.num_units;
    kp.workers = sch.workers;
    kp.sk_tile0 = sch.sk_tile0;
    kp.sk_iters = sch.sk_iters;
    kp.nseg_max = sch.nseg_max;
    kp.sk_slot_base = sch.sk_slot_base;
    kp.tail_tile0 = sch.tail_tile0;
    kp.tail_split = sch.tail_split;
    if (cb.tma && sch.tail_split > 1 && !(cb.mn && !b_3d)) {
        // Tail pieces read B through a box of their own width (the 2-D N-major
        // form already reads one 64-column box per atom column).
        const int piece = bcols / sch.tail_split;
        const bool ok = b_3d ? encode_3d_mn(&kp.tmB2, kp.B, b_mn_ext, a.K, a.K == 1 ? round_up(2 * Nv, 16) : 2 * kp.b_sk,
                                            static_cast<uint32_t>(piece / 64), nb_b, bst_b)
                             : encode_2d(&kp.tmB2, kp.B, a.K, Nv, Nv == 1 ? round_up(2 * a.K, 16) : 2 * kp.b_sn, 64,
                                         static_cast<uint32_t>(piece), nb_b, bst_b);
        if (!ok) return GEMM_F16_ERR_LAUNCH;
    }
    // Raster panel (tile rows whose tiles run side by side): 8 by default;
    // launches of at most four waves of tiles take 2, which measured 2 % faster
    // on 4096^3 (wider panels measured faster from 6144^3 up).  So do launches
    // with at most 16 tile columns (e.g. the MoE shape's 8): there a panel of 8
    // tile rows spreads each A row panel's tiles over two waves, and the second
    // wave re-reads it from HBM (131072 x 2048 x 7168: 4.71 GB of DRAM reads
    // with panels of 8, 3.65 GB with panels of 2, the same time).
    const int default_panel =
        (tiles <= 4 * static_cast<int64_t>(sch.workers) || tiles_n <= 16) ? 2 : 8;
    kp.panel = static_cast<int>(panel > 0 ? panel : default_panel);
    kp.BN = BN, kp.stages = stages;
    kp.a_flags = (ca.tma ? gemm_f16_dev::kOpTma : 0u) | (ca.mn ? gemm_f16_dev::kOpMnMajor : 0u) |
                 (a_3d ? gemm_f16_dev::kOpBox3d : 0u);
    kp.b_flags = (cb.tma ? gemm_f16_dev::kOpTma : 0u) | (cb.mn ? gemm_f16_dev::kOpMnMajor : 0u) |
                 (b_3d ? gemm_f16_dev::kOpBox3d : 0u);
    kp.c_tma = c_tma ? 1u : 0u;
    kp.c_stage = c_stage ? 1u : 0u;
    // Debug bounds check: the byte range each kernel view spans, every problem or
    // group included.  Value 2 is the checker's own test: each range ends 16
    // bytes early, so accesses to the last 8 elements are reported (and skipped)
    // although they are inside the real view.
    const int64_t dbg = opt(GEMM_F16_OPT_DEBUG_BOUNDS);
    kp.debug_bounds = dbg > 0 ? 1u : 0u;
    if (dbg > 0) {
        auto span = [&](int which, const void* ptr, int64_t rows, int64_t cols, int64_t s_r, int64_t s_c,
                        int64_t nb, int64_t bs) {
            int64_t e = 0;
            if (!view_extent(rows, cols, s_r, s_c, &e)) e = 0;
            if (nb > 1 && bs > 0 && !batch_extent(e, nb, bs, &e)) e = 0;
            kp.span_lo[which] = reinterpret_cast<uintptr_t>(ptr);
            kp.span_hi[which] = kp.span_lo[which] + static_cast<uintptr_t>(2 * e) - (dbg == 2 ? 16u : 0u);
        };
        const int64_t nb = (batched || grouped) ? a.batch : 1;
        span(gemm_f16_dev::kSpanA, kp.A, Mv, a.K, kp.a_sm, kp.a_sk, batched ? nb : 1, a_bs);
        span(gemm_f16_dev::kSpanB, kp.B, a.K, Nv, kp.b_sk, kp.b_sn, nb, b_bs);
        if (gated) span(gemm_f16_dev::kSpanBu, kp.Bu, a.K, Nv, kp.b_sk, kp.b_sn, nb, b_bs);
        span(gemm_f16_dev::kSpanC, kp.C, Mv, Nv, kp.c_sm, kp.c_sn, batched ? nb : 1, c_bs);
    }
    kp.test_stall = opt(GEMM_F16_OPT_TEST_STALL) == 1 ? 1u : 0u;
    // L2 eviction policies of the copies (kernel view): option 1 none, 2 evict
    // first, 3 evict last, 0 the default.  By default a one-problem launch of
    // several waves whose A' streams through L2 (at least 256 MB, twice the
    // L2), whose B' is small enough to stay there for the whole launch (at
    // most 48 MB: every tile row reads all of it) and whose raster runs each
    // A' row panel's tiles within one wave (panels of at most 2 tile rows, at
    // most 16 tile columns) marks A' evict-first (its rows are read by the
    // tiles of one raster row and then never again), B' evict-last, and the C
    // stores evict-first (written once, never read here), so that streaming
    // A' and C do not push B' out.  Measured on 131072 x 2048 x 7168: DRAM
    // reads 3.65 -> 2.14 GB per call (1.09 x the algorithmic bytes with C),
    // 1781 -> 1842 TFLOP/s back to back.  Batched and grouped launches, whose
    // problems each bring their own B', and shapes whose A' fits in L2 (4096^3)
    // measured 2-4 % slower with it, so they take no policy.
    const double a_stream = 2.0 * static_cast<double>(Mv) * static_cast<double>(a.K);
    const double b_resident = 2.0 * static_cast<double>(a.K) * static_cast<double>(Nv) * (gated ? 2.0 : 1.0);
    const bool streaming = !batched && !grouped && !gated && kp.panel <= 2 && tiles_n <= 16 && a_stream >= 256e6 &&
                           b_resident <= 48e6 && tiles >= 2 * static_cast<int64_t>(sch.workers);
    auto l2_kind = [](int64_t o, uint32_t dflt) { return o == 1 ? 0u : (o == 2 ? 1u : (o == 3 ? 2u : dflt)); };
    kp.l2_a = l2_kind(opt(GEMM_F16_OPT_L2_A), streaming ? 1u : 0u);
    kp.l2_b = l2_kind(opt(GEMM_F16_OPT_L2_B), streaming ? 2u : 0u);
    kp.l2_c = l2_kind(opt(GEMM_F16_OPT_L2_C), streaming ? 1u : 0u);
    kp.epi_smem = epi > 0 ? 1u : 0u;
    pl->fused = a.fused;
    if (a.fused) {
        kp.bias = static_cast<const __half*>(a.bias);
        kp.bias_up = static_cast<const __half*>(a.bias_up);
        kp.bias_bs = a.sbias;
        kp.act = a.act;
        kp.gated = gated ? 1 : 0;
        kp.bias_rows = swap ? 1 : 0;   // C^T: the bias runs along the kernel view's rows
    }
    // Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B fp16
    // (bits 7-9, 10-12 = 0), A/B MN-major flags (bits 15, 16), N >> 3 (bits
    // 17-22), M >> 4 (bits 24-28); M is 256 for the pair form.
    kp.idesc = (1u << 4) | ((ca.mn ? 1u : 0u) << 15) | ((cb.mn ? 1u : 0u) << 16) |
               ((static_cast<uint32_t>(BN) >> 3) << 17) | ((static_cast<uint32_t>(tile_rows) >> 4) << 24);
    kp.stage_b_bytes = stage_b;
    // (with both operands by TMA, the A' and B' issuers each arrive on the full barrier)
    if (pair) {
        kp.tx_bytes = 2u * stage_bytes;   // both CTAs' boxes complete on the leader's barrier
        kp.full_count = 2u;
    } else if (ca.tma && cb.tma) {
        kp.tx_bytes = gemm_f16_dev::kStageABytes + stage_b;
        kp.full_count = 2u;
    } else {
        kp.tx_bytes = (ca.tma ? gemm_f16_dev::kStageABytes : 0u) + (cb.tma ? stage_b : 0u);
        kp.full_count = ((ca.tma || cb.tma) ? 1u : 0u) +
                        ((!ca.tma || !cb.tma) ? static_cast<uint32_t>(gemm_f16_dev::kProducerThreads) : 0u);
    }

    pub.swap_ab = swap;
    pub.pair = pair;
    pub.cluster_ctas = cluster_ctas;
    pub.a_tma = ca.tma, pub.a_mn_major = ca.mn, pub.b_tma = cb.tma, pub.b_mn_major = cb.mn, pub.c_tma = c_tma;
    pub.a_box3d = a_3d && ca.tma, pub.b_box3d = b_3d && cb.tma;
    pub.tile_m = tile_rows, pub.tile_n = out_cols, pub.tiles_m = tiles_m, pub.tiles_n = tiles_n;
    pub.fused = a.fused ? 1 : 0;
    pub.gated = gated ? 1 : 0;
    pub.repack = repacked;
    pub.two_k_loads = static_cast<int>(kp.k2);
    pub.splits = splits, pub.kblocks = kblocks, pub.grid = grid;
    pub.units = static_cast<int>(tiles * splits);
    pub.streamk_tiles = sch.sk_iters > 0 ? static_cast<int>(tiles - sch.sk_tile0) : 0;
    pub.tail_split = sch.tail_split;
    pub.stages = stages, pub.smem_bytes = smem;
    pub.workspace_bytes = sch.partial_slots > 0
                              ? workspace_bytes_for(sch.partial_slots, BN, tiles, pair ? 2 : 1, &pl->counter_bytes,
                                                    &pl->partial_bytes)
                              : 0;
    return GEMM_F16_OK;
}

gemm_f16_status launch(Plan& pl, DevInfo& dev, float* partials, int* counters, cudaStream_t stream)
{
    KernelParams& kp = pl.kp;
    kp.ws = partials;
    kp.counters = counters;
    if (pl.pub.grid == 0) return GEMM_F16_OK;   // no tile (every group empty)
    if (!set_smem_attributes(dev)) return GEMM_F16_ERR_LAUNCH;
    // Every launch is a programmatic dependent of the kernel before it on the
    // stream (unless GEMM_F16_OPT_PDL = 1): its prologue may overlap that
    // kernel's tail, and the kernels wait (griddepcontrol.wait) before their
    // first global-memory access.
    const bool pdl = opt(GEMM_F16_OPT_PDL) != 1;
    auto config = [&](cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, unsigned grid, unsigned block, size_t smem,
                      int cluster) {
        cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(block);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        int n = 0;
        if (cluster > 1) {
            attr[n].id = cudaLaunchAttributeClusterDimension;
            attr[n].val.clusterDim.x = cluster;
            attr[n].val.clusterDim.y = 1;
            attr[n].val.clusterDim.z = 1;
            ++n;
        }
        if (pdl) {
            attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[n].val.programmaticStreamSerializationAllowed = 1;
            ++n;
        }
        cfg.attrs = attr;
        cfg.numAttrs = n;
    };
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    if (pl.ncopies > 0) {   // every copy in one launch, before the GEMM on the same stream
        gemm_f16_dev::RepackBatch rb;
        rb.n = pl.ncopies;
        int64_t items = 0;
        for (int i = 0; i < pl.ncopies; ++i) {
            rb.c[i] = pl.copies[i];
            items += gemm_f16_dev::repack_items(pl.copies[i]);
        }
        config(cfg, attr, copy_blocks(items, dev.sms, gemm_f16_dev::kRepackBlocksPerSm), gemm_f16_dev::kRepackThreads, 0,
               1);
        if (cudaLaunchKernelEx(&cfg, gemm_f16_dev::repack_rows, rb) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_F16_ERR_LAUNCH;
        }
    }
    const bool multi = kp.gmode != 0;
    config(cfg, attr, static_cast<unsigned>(pl.pub.grid), gemm_f16_dev::kNumThreads, pl.pub.smem_bytes,
           pl.pub.pair ? pl.pub.cluster_ctas : 1);
    using gemm_f16_dev::gemm_f16_persistent;
    const cudaError_t e =
        !pl.pub.pair ? (pl.fused ? cudaLaunchKernelEx(&cfg, gemm_f16_persistent<false, true, true>, kp)
                        : multi  ? cudaLaunchKernelEx(&cfg, gemm_f16_persistent<false, true>, kp)
                                 : cudaLaunchKernelEx(&cfg, gemm_f16_persistent<false, false>, kp))
        : pl.fused ? cudaLaunchKernelEx(&cfg, gemm_f16_persistent<true, true, true>, kp)
        : multi    ? cudaLaunchKernelEx(&cfg, gemm_f16_persistent<true, true>, kp)
                   : cudaLaunchKernelEx(&cfg, gemm_f16_persistent<true, false>, kp);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_F16_ERR_LAUNCH;
    }
    if (pl.unpack) {   // C from the aligned buffer into place, after the GEMM on the same stream
        config(cfg, attr, copy_blocks(gemm_f16_dev::unpack_items(pl.out), dev.sms, gemm_f16_dev::kUnpackBlocksPerSm),
               gemm_f16_dev::kRepackThreads, 0, 1);
        if (cudaLaunchKernelEx(&cfg, gemm_f16_dev::unpack_rows, pl.out) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_F16_ERR_LAUNCH;
        }
    }
    if (cudaGetLastError() != cudaSuccess) return GEMM_F16_ERR_LAUNCH;
    return GEMM_F16_OK;
}

// Grow one buffer of the library workspace.  Earlier calls may still use the
// old buffer, so the device is synchronised before it is freed.
bool grow(void** buf, size_t* have, size_t need, bool zero, cudaStream_t stream)
{
    if (*have >= need) return true;
    if (*buf) {
        cudaDeviceSynchronize();
        cudaFree(*buf);
        *buf = nullptr;
        *have = 0;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, need) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (zero && cudaMemsetAsync(p, 0, need, stream) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p);
        return false;
    }
    *buf = p;
    *have = need;
    return true;
}

void* repack_buffer(size_t bytes, bool plan_only, cudaStream_t stream)
{
    if (plan_only) return reinterpret_cast<void*>(uintptr_t(1) << 21);
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mutex);
    Workspace& w = g_ws[d];
    if (!grow(&w.repack, &w.repack_bytes, bytes, false, stream)) return nullptr;
    return w.repack;
}

gemm_f16_status run(const Args& args, void* user_ws, size_t user_ws_bytes, bool use_library_ws, cudaStream_t stream)
{
    Args a = args;
    a.repack = use_library_ws;
    DevInfo* dev = nullptr;
    gemm_f16_status st = validate(a, true, &dev);
    if (st != GEMM_F16_OK) return st;
    Plan pl;
    st = make_plan(a, *dev, &pl, false, stream);
    if (st != GEMM_F16_OK) return st;
    float* partials = nullptr;
    int* counters = nullptr;
    if (pl.pub.workspace_bytes > 0) {
        if (use_library_ws) {
            int d = 0;
            cudaGetDevice(&d);
            std::lock_guard<std::mutex> lk(g_mutex);
            Workspace& w = g_ws[d];
            void* c = w.counters;
            if (!grow(&w.partials, &w.partial_bytes, pl.partial_bytes, false, stream) ||
                !grow(&c, &w.counter_bytes, pl.counter_bytes, true, stream))
                return GEMM_F16_ERR_OUT_OF_MEMORY;
            w.counters = static_cast<int*>(c);
            partials = static_cast<float*>(w.partials);
            counters = w.counters;
        } else {
            if (!user_ws || user_ws_bytes < pl.pub.workspace_bytes || (reinterpret_cast<uintptr_t>(user_ws) & 255u))
                return GEMM_F16_ERR_OUT_OF_MEMORY;
            // A caller's workspace may hold anything (another shape's partials):
            // clear the counter block on the stream before the kernel.
            counters = static_cast<int*>(user_ws);
            partials = reinterpret_cast<float*>(static_cast<char*>(user_ws) + pl.counter_bytes);
            if (cudaMemsetAsync(counters, 0, pl.counter_bytes, stream) != cudaSuccess) {
                cudaGetLastError();
                return GEMM_F16_ERR_LAUNCH;
            }
        }
    }
    return launch(pl, *dev, partials, counters, stream);
}

// ---------------------------------------------------------------------------
// Fixed scratch for gemm_f16_noalloc(): the split-K / stream-K counters and
// partial sums live in this file-scope device array instead of memory the
// library allocates.  Every device that loads the library holds it (8 MiB)
// until the process exits.  In host code `g_noalloc_scratch` is only a
// stand-in for the symbol, never a device address: the address comes from
// cudaGetSymbolAddress, taken once per device with that device current.
constexpr size_t kNoAllocScratchBytes = GEMM_F16_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The address is cached per device together with the context it was taken in:
// after cudaDeviceReset (or anything else that replaces the device's primary
// context) the module is loaded again at another address, so a call in a new
// context looks the address up again instead of using a stale one.
struct NoAllocScratch {
    void* ptr = nullptr;
    CUcontext ctx = nullptr;
};
NoAllocScratch g_noalloc[kMaxDevices];

// Device address of the scratch array on the current device (nullptr if the
// runtime could not provide it).
void* noalloc_scratch()
{
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    load_entry_points();
    CUcontext ctx = nullptr;
    if (!g_ctx_current || g_ctx_current(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    std::lock_guard<std::mutex> lk(g_mutex);
    NoAllocScratch& e = g_noalloc[d];
    if (!e.ptr || !ctx || e.ctx != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        // (the lookup makes the primary context current if it was not yet)
        if (!g_ctx_current || g_ctx_current(&ctx) != CUDA_SUCCESS) ctx = nullptr;
        e.ptr = p;
        e.ctx = ctx;
    }
    return e.ptr;
}

gemm_f16_status run_noalloc(const Args& a, cudaStream_t stream)
{
    DevInfo* dev = nullptr;
    gemm_f16_status st = validate(a, true, &dev);
    if (st != GEMM_F16_OK) return st;
    Plan pl;
    st = make_plan(a, *dev, &pl);
    if (st != GEMM_F16_OK) return st;
    float* partials = nullptr;
    int* counters = nullptr;
    if (pl.pub.workspace_bytes > 0) {
        if (pl.pub.workspace_bytes > kNoAllocScratchBytes) return GEMM_F16_ERR_OUT_OF_MEMORY;
        void* s = noalloc_scratch();
        if (!s) return GEMM_F16_ERR_LAUNCH;
        counters = static_cast<int*>(s);
        partials = reinterpret_cast<float*>(static_cast<char*>(s) + pl.counter_bytes);
        // The array keeps the previous call's contents; the counters must start
        // at zero (the partials are always written before they are read).
        if (cudaMemsetAsync(counters, 0, pl.counter_bytes, stream) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_F16_ERR_LAUNCH;
        }
    }
    return launch(pl, *dev, partials, counters, stream);
}

void set_fused(Args& a, const void* B_up, const void* bias, const void* bias_up, int64_t stride_bias, int act)
{
    a.fused = true;
    a.Bu = B_up;
    a.bias = bias;
    a.bias_up = bias_up;
    a.sbias = stride_bias;
    a.act = act;
}

// Sum of the group rows (false if one is negative or the sum overflows).
bool total_rows(const int64_t* group_rows, int64_t groups, int64_t* total)
{
    if (!group_rows || groups < 1 || groups > gemm_f16_dev::kMaxGroups) return false;
    int64_t t = 0;
    for (int64_t g = 0; g < groups; ++g)
        if (group_rows[g] < 0 || __builtin_add_overflow(t, group_rows[g], &t)) return false;
    *total = t;
    return true;
}

}  // namespace

extern "C" {

gemm_f16_status gemm_f16(const void* A, int64_t stride_am, int64_t stride_ak, const void* B, int64_t stride_bk,
                         int64_t stride_bn, void* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                         cudaStream_t stream)
{
    const Args a{A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K};
    return run(a, nullptr, 0, true, stream);
}

gemm_f16_status gemm_f16_ws(const void* A, int64_t stride_am, int64_t stride_ak, const void* B, int64_t stride_bk,
                            int64_t stride_bn, void* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    const Args a{A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K};
    return run(a, workspace, workspace_bytes, false, stream);
}

gemm_f16_status gemm_f16_noalloc(const void* A, int64_t stride_am, int64_t stride_ak, const void* B,
                                 int64_t stride_bk, int64_t stride_bn, void* C, int64_t ldc, int64_t M, int64_t N,
                                 int64_t K, cudaStream_t stream)
{
    const Args a{A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K};
    return run_noalloc(a, stream);
}

gemm_f16_status gemm_f16_batched(const void* A, int64_t stride_ab, int64_t stride_am, int64_t stride_ak,
                                 const void* B, int64_t stride_bb, int64_t stride_bk, int64_t stride_bn, void* C,
                                 int64_t stride_cb, int64_t ldc, int64_t M, int64_t N, int64_t K, int64_t batch,
                                 cudaStream_t stream)
{
    Args a{A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K};
    a.batch = batch;
    a.sab = stride_ab, a.sbb = stride_bb, a.scb = stride_cb;
    return run(a, nullptr, 0, true, stream);
}

gemm_f16_status gemm_f16_grouped(const void* A, int64_t stride_am, int64_t stride_ak, const void* B,
                                 int64_t stride_bg, int64_t stride_bk, int64_t stride_bn, void* C, int64_t ldc,
                                 const int64_t* group_rows, int64_t groups, int64_t N, int64_t K,
                                 cudaStream_t stream)
{
    int64_t total = 0;
    if (!total_rows(group_rows, groups, &total)) return GEMM_F16_ERR_INVALID_VALUE;
    if (total == 0) return (A && B && C && N > 0 && K > 0) ? GEMM_F16_OK : GEMM_F16_ERR_INVALID_VALUE;
    Args a{A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, total, N, K};
    a.batch = groups;
    a.sbb = stride_bg;
    a.rows = group_rows;
    return run(a, nullptr, 0, true, stream);
}

gemm_f16_status gemm_f16_fused(const void* A, int64_t stride_am, int64_t stride_ak, const void* B, int64_t stride_bk,
                               int64_t stride_bn, const void* B_up, const void* bias, const void* bias_up, int act,
                               void* C, int64_t ldc, int64_t M, int64_t N, int64_t K, cudaStream_t stream)
{
    Args a{A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K};
    set_fused(a, B_up, bias, bias_up, 0, act);
    return run(a, nullptr, 0, true, stream);
}

gemm_f16_status gemm_f16_batched_fused(const void* A, int64_t stride_ab, int64_t stride_am, int64_t stride_ak,
                                       const void* B, int64_t stride_bb, int64_t stride_bk, int64_t stride_bn,
                                       const void* B_up, const void* bias, const void* bias_up, int64_t stride_bias,
                                       int act, void* C, int64_t stride_cb, int64_t ldc, int64_t M, int64_t N,
                                       int64_t K, int64_t batch, cudaStream_t stream)
{
    Args a{A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K};
    a.batch = batch;
    a.sab = stride_ab, a.sbb = stride_bb, a.scb = stride_cb;
    set_fused(a, B_up, bias, bias_up, stride_bias, act);
    return run(a, nullptr, 0, true, stream);
}

gemm_f16_status gemm_f16_grouped_fused(const void* A, int64_t stride_am, int64_t stride_ak, const void* B,
                                       int64_t stride_bg, int64_t stride_bk, int64_t stride_bn, const void* B_up,
                                       const void* bias, const void* bias_up, int64_t stride_bias, int act, void* C,
                                       int64_t ldc, const int64_t* group_rows, int64_t groups, int64_t N, int64_t K,
                                       cudaStream_t stream)
{
    int64_t total = 0;
    if (!total_rows(group_rows, groups, &total)) return GEMM_F16_ERR_INVALID_VALUE;
    if (act < GEMM_F16_ACT_NONE || act > GEMM_F16_ACT_GELU || stride_bias < 0 || (bias_up && !B_up))
        return GEMM_F16_ERR_INVALID_VALUE;
    if (total == 0) return (A && B && C && N > 0 && K > 0) ? GEMM_F16_OK : GEMM_F16_ERR_INVALID_VALUE;
    Args a{A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, total, N, K};
    a.batch = groups;
    a.sbb = stride_bg;
    a.rows = group_rows;
    set_fused(a, B_up, bias, bias_up, stride_bias, act);
    return run(a, nullptr, 0, true, stream);
}

gemm_f16_status gemm_f16_fused_get_plan(const void* A, int64_t stride_am, int64_t stride_ak, const void* B,
                                        int64_t stride_bk, int64_t stride_bn, const void* B_up, const void* bias,
                                        const void* bias_up, int act, void* C, int64_t ldc, int64_t M, int64_t N,
                                        int64_t K, gemm_f16_plan* plan)
{
    if (!plan) return GEMM_F16_ERR_INVALID_VALUE;
    Args a{A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K};
    set_fused(a, B_up, bias, bias_up, 0, act);
    a.repack = true;
    DevInfo* dev = nullptr;
    gemm_f16_status st = validate(a, true, &dev);
    if (st != GEMM_F16_OK) return st;
    Plan pl;
    st = make_plan(a, *dev, &pl, true);
    if (st == GEMM_F16_OK) *plan = pl.pub;
    return st;
}

gemm_f16_status gemm_f16_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes)
{
    if (!bytes || M <= 0 || N <= 0 || K <= 0) return GEMM_F16_ERR_INVALID_VALUE;
    DevInfo* dev = nullptr;
    gemm_f16_status st = device_info(&dev);
    if (st != GEMM_F16_OK) return st;
    bool swap;
    int64_t Mv, Nv;
    int BN, tiles_m, tiles_n, kblocks, splits;
    shape_plan(M, N, K, dev->sms, true, &swap, &Mv, &Nv, &BN, &tiles_m, &tiles_n, &kblocks, &splits);
    // The plan also depends on the operands' layout (single or pair form), so
    // report the larger of the two requirements.
    size_t need = 0;
    for (int pair = 0; pair < 2; ++pair) {
        const int64_t rows = pair ? 2 * gemm_f16_dev::kBM : gemm_f16_dev::kBM;
        const int64_t tiles = ((Mv + rows - 1) / rows) * tiles_n;
        const int workers = pair ? std::max(1, dev->sms / 2) : dev->sms;
        // the single form may gather an operand, and the swapped form (single or
        // pair) has fewer tiles than SMs: both turn stream-K on by default
        const int64_t sk = opt(GEMM_F16_OPT_STREAMK);
        const int sp = splits == 1 ? kseg_default(swap, pair != 0, false, tiles, kblocks, dev->sms) : splits;
        const bool streamk = sp == 1 && (sk == 2 || (sk == 0 && (!pair || swap)));
        const Schedule s = make_schedule(tiles, kblocks, sp, workers, BN, pair ? 128 : 64, streamk);
        if (s.partial_slots > 0)
            need = std::max(need, workspace_bytes_for(s.partial_slots, BN, tiles, pair ? 2 : 1, nullptr, nullptr));
    }
    *bytes = need;
    return GEMM_F16_OK;
}

const char* gemm_f16_status_string(int status)
{
    switch (status) {
    case GEMM_F16_OK: return "GEMM_F16_OK";
    case GEMM_F16_ERR_INVALID_VALUE: return "GEMM_F16_ERR_INVALID_VALUE";
    case GEMM_F16_ERR_ALIAS: return "GEMM_F16_ERR_ALIAS";
    case GEMM_F16_ERR_UNSUPPORTED_DEVICE: return "GEMM_F16_ERR_UNSUPPORTED_DEVICE";
    case GEMM_F16_ERR_OUT_OF_MEMORY: return "GEMM_F16_ERR_OUT_OF_MEMORY";
    case GEMM_F16_ERR_LAUNCH: return "GEMM_F16_ERR_LAUNCH";
    case GEMM_F16_ERR_TIMEOUT: return "GEMM_F16_ERR_TIMEOUT";
    case GEMM_F16_ERR_BOUNDS: return "GEMM_F16_ERR_BOUNDS";
    default: return "GEMM_F16_UNKNOWN_STATUS";
    }
}

gemm_f16_status gemm_f16_device_status(int* status, int reset)
{
    if (!status) return GEMM_F16_ERR_INVALID_VALUE;
    DevInfo* dev = nullptr;
    gemm_f16_status st = device_info(&dev);
    if (st != GEMM_F16_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return GEMM_F16_ERR_LAUNCH;
    }
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_f16_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_F16_ERR_LAUNCH;
    }
    *status = v;
    if (reset) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_gemm_f16_status, &zero, sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_F16_ERR_LAUNCH;
        }
        int d = 0;
        cudaGetDevice(&d);
        std::lock_guard<std::mutex> lk(g_mutex);
        if (g_ws[d].counters && cudaMemset(g_ws[d].counters, 0, g_ws[d].counter_bytes) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_F16_ERR_LAUNCH;
        }
    }
    return GEMM_F16_OK;
}

gemm_f16_status gemm_f16_get_plan(const void* A, int64_t stride_am, int64_t stride_ak, const void* B,
                                  int64_t stride_bk, int64_t stride_bn, void* C, int64_t ldc, int64_t M, int64_t N,
                                  int64_t K, gemm_f16_plan* plan)
{
    if (!plan) return GEMM_F16_ERR_INVALID_VALUE;
    Args a{A, stride_am, stride_ak, B, stride_bk, stride_bn, C, ldc, M, N, K};
    a.repack = true;   // as gemm_f16() would run it
    DevInfo* dev = nullptr;
    gemm_f16_status st = validate(a, true, &dev);
    if (st != GEMM_F16_OK) return st;
    Plan pl;
    st = make_plan(a, *dev, &pl, true);
    if (st == GEMM_F16_OK) *plan = pl.pub;
    return st;
}

gemm_f16_status gemm_f16_set_option(int option, int64_t value)
{
    // (12 is not an option: that number is left unused)
    if (option < 1 || option > 20 || option == 12 || value < 0) return GEMM_F16_ERR_INVALID_VALUE;
    if (option == GEMM_F16_OPT_TWO_K_LOADS && value > 1) return GEMM_F16_ERR_INVALID_VALUE;
    if ((option == GEMM_F16_OPT_L2_A || option == GEMM_F16_OPT_L2_B || option == GEMM_F16_OPT_L2_C) && value > 3)
        return GEMM_F16_ERR_INVALID_VALUE;
    if (option == GEMM_F16_OPT_DEBUG_BOUNDS && value > 2) return GEMM_F16_ERR_INVALID_VALUE;
    if (option == GEMM_F16_OPT_PDL && value > 1) return GEMM_F16_ERR_INVALID_VALUE;
    if (option == GEMM_F16_OPT_TEST_STALL && value > 1) return GEMM_F16_ERR_INVALID_VALUE;
    if (option == GEMM_F16_OPT_REPACK && value > 2) return GEMM_F16_ERR_INVALID_VALUE;
    if (option == GEMM_F16_OPT_MAX_STAGES && value == 1) return GEMM_F16_ERR_INVALID_VALUE;
    if (option == GEMM_F16_OPT_TAIL_SPLIT && value > 1) return GEMM_F16_ERR_INVALID_VALUE;
    if (option == GEMM_F16_OPT_STREAMK && value > 2) return GEMM_F16_ERR_INVALID_VALUE;
    if (option == GEMM_F16_OPT_PAIR && value > 2) return GEMM_F16_ERR_INVALID_VALUE;
    if (option == GEMM_F16_OPT_FORCE_GATHER && value > 7) return GEMM_F16_ERR_INVALID_VALUE;
    if (option == GEMM_F16_OPT_TILE_N && value != 0 && (value % 64 != 0 || value > 256))
        return GEMM_F16_ERR_INVALID_VALUE;
    if (option == GEMM_F16_OPT_SWAP && value > 2) return GEMM_F16_ERR_INVALID_VALUE;
    g_opt[option].store(value, std::memory_order_relaxed);
    return GEMM_F16_OK;
}

int gemm_f16_abi_version(void) { return GEMM_F16_ABI_VERSION; }

}  // extern "C"
