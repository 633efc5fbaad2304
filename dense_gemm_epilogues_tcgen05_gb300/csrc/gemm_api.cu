// gemm_api.cu -- host side of the C ABI declared in include/gemm_gb300.h:
// argument validation, the choice of kernel family, TMA tensor-map encoding
// for each operand along its contiguous dimension, launch geometry and the
// device status word.
//
// The stride convention follows "Case Study: Steel's BlockMMA" (transposition
// carried only by the A_str_m / A_str_k style stride constants); the launch
// geometry replaces the one-threadgroup-per-tile grid of "X3: Metal GEMM"
// section 6 by a persistent grid of at most one CTA per SM walking tiles.
#include <cuda.h>
#include <cuda_runtime_api.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <iterator>
#include <mutex>

#include "../../include/gemm_gb300.h"
#include "kernel_args.h"

// Device status word: kernels OR status bits into it; gemm_device_status reads
// and clears it.
__device__ unsigned int g_gemm_status_word;

namespace {

using namespace gb300;

constexpr int kMaxDevices = 64;

int elem_bytes(int dt) { return dt == GEMM_F32 ? 4 : (dt == GEMM_E4M3 ? 1 : 2); }

bool valid_dtype(int dt) { return dt >= GEMM_F32 && dt <= GEMM_E4M3; }

// ----------------------------------------------------- driver entry points --

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*AddrRangeFn)(CUdeviceptr *, size_t *, CUdeviceptr);
typedef CUresult (*PtrAttrFn)(void *, CUpointer_attribute, CUdeviceptr);

struct DriverFns {
    EncodeTiledFn encode = nullptr;
    AddrRangeFn addr_range = nullptr;
    PtrAttrFn ptr_attr = nullptr;  // optional: extents of host allocations
    bool ok = false;
};

const DriverFns &driver_fns() {
    static DriverFns fns;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.encode = reinterpret_cast<EncodeTiledFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.addr_range = reinterpret_cast<AddrRangeFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.ptr_attr = reinterpret_cast<PtrAttrFn>(p);
        fns.ok = fns.encode != nullptr && fns.addr_range != nullptr;
    });
    return fns;
}

// ------------------------------------------------------- per-device state --

struct DeviceState {
    bool ready = false;
    int ordinal = -1;
    int num_sms = 0;
    unsigned int *status = nullptr;
    // Resident clusters of the pair kernel by (cluster of 2 or 4 CTAs, ab incl.
    // 3xTF32, out); -1 = not queried yet.
    int max_clusters[2][5][4];
};

std::mutex g_dev_mu;
DeviceState g_dev[kMaxDevices];

// State of the current device; initialised on first use with that device current.
gemm_status_t device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            return GEMM_ERR_CUDA;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gemm_status_word) != cudaSuccess || p == nullptr) return GEMM_ERR_CUDA;
        d.ordinal = dev;
        d.num_sms = sms;
        d.status = static_cast<unsigned int *>(p);
        for (auto &plane : d.max_clusters)
            for (auto &row : plane)
                for (int &v : row) v = -1;
        d.ready = true;
    }
    *out = &d;
    return GEMM_OK;
}

// ------------------------------------------------------------- the plan --

struct Operand {
    bool tma = false;      // streamed by TMA
    bool mn_major = false; // the M (or N) index is the contiguous one
};

// Can the (rows x cols) operand with element strides (s_rows, s_cols) be
// described by a 2-D tensor map whose inner dimension is `cols` when
// k_inner, else `rows`?  `inner_stride` must be 1; the outer stride in bytes
// a multiple of 16 (unless the outer extent is 1); base 16-byte aligned.
bool tma_ok(const void *base, int64_t outer_extent, int64_t inner_stride, int64_t outer_stride, int es) {
    if (inner_stride != 1) return false;
    if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0) return false;
    if (outer_extent == 1) return true;
    const int64_t bytes = outer_stride * es;
    return bytes % 16 == 0 && bytes > 0 && bytes < (int64_t(1) << 40);
}

// An operand with logical shape (mn x k), element (i, k) at i*s_mn + k*s_k.
Operand plan_operand(const void *base, int64_t mn, int64_t k, int64_t s_mn, int64_t s_k, int es) {
    Operand o;
    if (tma_ok(base, mn, s_k, s_mn, es)) {
        o.tma = true;
        o.mn_major = false;
    } else if (tma_ok(base, k, s_mn, s_k, es)) {
        o.tma = true;
        o.mn_major = true;
    }
    return o;
}

struct Plan {
    gemm_path_t path = GEMM_PATH_NOOP;
    Operand a, b;
};

gemm_status_t make_plan(int64_t M, int64_t N, int64_t K, int ab, const void *A, int64_t sam, int64_t sak,
                        const void *B, int64_t sbk, int64_t sbn, const void *C, int64_t ldc, int cd, float alpha,
                        const float *bias, int epi, Plan *plan, bool fp8_out = false) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (!valid_dtype(ab) || !valid_dtype(cd)) return GEMM_ERR_INVALID_ARG;
    if (epi < GEMM_EPI_NONE || epi > GEMM_EPI_BIAS_RELU) return GEMM_ERR_INVALID_ARG;
    if (cd == GEMM_E4M3 && !fp8_out) return GEMM_ERR_UNSUPPORTED;
    if (ab == GEMM_F32 && cd != GEMM_F32) return GEMM_ERR_UNSUPPORTED;
    if (ab == GEMM_E4M3 && cd == GEMM_F16) return GEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) {
        plan->path = GEMM_PATH_NOOP;
        return GEMM_OK;
    }
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
    if (C == nullptr || ldc < N) return GEMM_ERR_INVALID_ARG;
    if (epi != GEMM_EPI_NONE && bias == nullptr) return GEMM_ERR_INVALID_ARG;
    if (K == 0 || alpha == 0.0f) {
        plan->path = GEMM_PATH_EPILOGUE_ONLY;
        return GEMM_OK;
    }
    if (A == nullptr || B == nullptr) return GEMM_ERR_INVALID_ARG;
    if (sam < 0 || sak < 0 || sbk < 0 || sbn < 0) return GEMM_ERR_INVALID_ARG;
    if (ab == GEMM_F32) {
        plan->path = GEMM_PATH_SIMT;
        return GEMM_OK;
    }
    const int es = elem_bytes(ab);
    plan->a = plan_operand(A, M, K, sam, sak, es);
    plan->b = plan_operand(B, N, K, sbn, sbk, es);
    const int64_t tiles = ((M + 127) / 128) * ((N + 127) / 128);
    plan->path = (plan->a.tma && plan->b.tma && tiles < INT32_MAX) ? GEMM_PATH_TCGEN05 : GEMM_PATH_SIMT;
    return GEMM_OK;
}

// ------------------------------------------------------- pointer checks --

// The byte range [p, p + bytes) must lie inside one allocation the device can
// address: device memory, or pinned / managed host memory.  Plain pageable
// host pointers are rejected: a kernel given one would fault.  Where the
// driver reports the allocation's extent (device memory always; host
// allocations where it knows them) the range must fit inside it.  When
// `local` is given it is set to whether the range is device memory of the
// device `ordinal` (the current one) -- the only memory a multicast tensor
// map may cover.
gemm_status_t check_range(const void *p, size_t bytes, int ordinal = -1, bool *local = nullptr) {
    if (local != nullptr) *local = false;
    if (bytes == 0) return GEMM_OK;
    if (p == nullptr) return GEMM_ERR_INVALID_ARG;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_INVALID_ARG;
    }
    if (attr.type == cudaMemoryTypeUnregistered) return GEMM_ERR_INVALID_ARG;
    const DriverFns &fns = driver_fns();
    CUdeviceptr base = 0;
    size_t size = 0;
    if (attr.type == cudaMemoryTypeDevice) {
        if (fns.addr_range(&base, &size, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS) size = 0;
    } else if (fns.ptr_attr != nullptr) {
        // pinned or managed host memory: its extent as the driver recorded it, if it did
        void *start = nullptr;
        if (fns.ptr_attr(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, reinterpret_cast<CUdeviceptr>(p)) !=
                CUDA_SUCCESS ||
            fns.ptr_attr(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS)
            size = 0;
        base = reinterpret_cast<CUdeviceptr>(start);
    }
    if (size > 0) {
        const uint64_t first = reinterpret_cast<uint64_t>(p);
        if (first < base || first + bytes > base + size) return GEMM_ERR_INVALID_ARG;
    }
    if (local != nullptr) *local = attr.type == cudaMemoryTypeDevice && attr.device == ordinal;
    return GEMM_OK;
}

size_t span_bytes(int64_t rows, int64_t cols, int64_t s_rows, int64_t s_cols, int es) {
    if (rows == 0 || cols == 0) return 0;
    return static_cast<size_t>(((rows - 1) * s_rows + (cols - 1) * s_cols + 1) * es);
}

// ------------------------------------------------------ tensor maps --

CUtensorMapDataType tma_dtype(int ab) {
    switch (ab) {
    case GEMM_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case GEMM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    default: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
    }
}

// 2-D map over (inner, outer) with a box of (box_inner, box_outer) elements,
// 128-byte swizzle, zero fill outside the tensor.
gemm_status_t encode_2d(CUtensorMap *map, int ab, const void *base, int64_t inner, int64_t outer,
                        int64_t outer_stride_elems, uint32_t box_inner, uint32_t box_outer) {
    const int es = elem_bytes(ab);
    int64_t stride_bytes = outer_stride_elems * es;
    if (outer == 1) stride_bytes = ((inner * es + 15) / 16) * 16;  // never used to address an element
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride_bytes)};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = driver_fns().encode(map, tma_dtype(ab), 2, const_cast<void *>(base), dims, strides, box, estr,
                                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// 2-D map with an explicit data type (3xTF32 arrays are plain fp32).
gemm_status_t encode_2d_dt(CUtensorMap *map, CUtensorMapDataType dt, int es, const void *base, int64_t inner,
                           int64_t outer, int64_t outer_stride_elems, uint32_t box_inner, uint32_t box_outer) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(outer_stride_elems * es)};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = driver_fns().encode(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// Map for an operand of logical shape (mn x k): K-major boxes are
// (k-block x tile rows); MN-major boxes are (one 128-byte swizzle row of MN x
// k-block), several per tile.
gemm_status_t encode_operand(CUtensorMap *map, int ab, const void *base, const Operand &o, int64_t mn, int64_t k,
                             int64_t s_mn, int64_t s_k, uint32_t tile_mn) {
    const uint32_t swz = 128u / elem_bytes(ab);
    if (!o.mn_major) return encode_2d(map, ab, base, k, mn, s_mn, swz, tile_mn);
    return encode_2d(map, ab, base, mn, k, s_k, swz, swz);
}

// Map of the output C (N x M, row pitch ldc) for the pair kernel's staged
// epilogue: boxes of 32 rows x 64 bytes with the 64-byte swizzle.  Returns
// false (and the kernel stores C directly) when C's base or row pitch rules
// out TMA.
bool encode_c(CUtensorMap *map, int cd, void *C, int64_t M, int64_t N, int64_t ldc) {
    const int es = elem_bytes(cd);
    const int64_t pitch = ldc * es;
    if ((reinterpret_cast<uintptr_t>(C) & 15u) != 0 || pitch % 16 != 0 || pitch <= 0 || pitch >= (int64_t(1) << 40))
        return false;
    const CUtensorMapDataType dt = cd == GEMM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : cd == GEMM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(64 / es), 32u};
    cuuint32_t estr[2] = {1, 1};
    return driver_fns().encode(map, dt, 2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ 3xTF32 --

// Stacked K-major hi/lo arrays of A (2M x pitch) and B (2N x pitch), pitch = K
// rounded up to 4 floats (16-byte rows for TMA), each array 256-byte aligned.
int64_t tf32x3_pitch(int64_t K) { return (K + 3) / 4 * 4; }
size_t round256(size_t x) { return (x + 255) / 256 * 256; }
size_t tf32x3_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || M >= (int64_t(1) << 30) || N >= (int64_t(1) << 30) || K > INT32_MAX)
        return 0;
    const size_t p = static_cast<size_t>(tf32x3_pitch(K));
    return round256(2 * static_cast<size_t>(M) * p * 4) + round256(2 * static_cast<size_t>(N) * p * 4);
}

// ------------------------------------------------------------ tile choice --

// Tuning settings (gemm_set_*): each thread has its own, so a test or tuning
// call in one thread never changes the kernel another thread's call runs.
struct Tuning {
    int tile_policy = GEMM_TILE_AUTO;
    int tile_policy_bn = 0;
    int schedule = GEMM_SCHED_AUTO;
    int operand_order = GEMM_ORDER_AUTO;
    int multicast = GEMM_MCAST_AUTO;
    int q4_kernel = GEMM_Q4_AUTO;
};
thread_local Tuning t_tuning;

std::atomic<unsigned int> g_epoch{0};

// The calling thread's last successful gemm() launch (gemm_last_launch).
thread_local gemm_launch_info_t t_last_launch = {};

gemm_status_t record(gemm_status_t st, const gemm_launch_info_t &info) {
    if (st == GEMM_OK) t_last_launch = info;
    return st;
}

// Stream-K workspace layout for `clusters` pairs: partial sums, then flags.
size_t partial_bytes(int clusters) { return static_cast<size_t>(clusters) * 2 * kPartialFloatsPerCta * 4; }
size_t workspace_bytes_for(int clusters) {
    return partial_bytes(clusters) + ((static_cast<size_t>(clusters) * kFlagsPerCluster * 4 + 255) / 256) * 256;
}

unsigned int next_epoch() {
    unsigned int e = g_epoch.fetch_add(1) + 1;
    if (e == 0) e = g_epoch.fetch_add(1) + 1;  // 0 means "not ready"
    return e;
}

// Schedule of the pair kernel: the tiles of the last one or two waves are
// split over all clusters by k-block ranges (stream-K), the rest are whole
// tiles, so every cluster ends at about the same time.  Measured on GB300 the
// balance gain is small (the GPU runs near its power limit, so the SMs left
// idle by a partial last wave let the busy ones clock up) and the fix-up
// epilogues cost a fixed time per split tile, so the automatic mode uses it
// only when (a) whole tiles alone would leave >= 10% of the cluster-time idle
// in the last wave, (b) tiles are long (>= 48 k-blocks) and (c) at least one
// wave of whole tiles remains for the fix-ups to hide behind.  Results:
// bf16 / fp16 4096^3 +2%; fp8 4096^3 (32 k-blocks) and M=8192 bias+GELU
// (3.8% idle) would lose 2-4% and keep whole tiles.  Stream-K always needs at
// least 8 k-blocks per cluster.
//
// Cut points of the stream-K range.  A cluster's piece ends with the first
// k-blocks of a tile (its OWNER segment) unless it ends on a tile boundary.
// When that segment is short and something precedes it in the piece, its MMAs
// finish before the epilogue of the segment before it has freed the other
// accumulator, and the next segment waits: measured on GB300 (fp16 4096^3) a
// 7-k-block OWNER after a whole tile cost 4 us, a tenth of the cluster's
// run.  So each piece is charged max(0, E - b) extra k-blocks for such an
// ending of b k-blocks (E: an epilogue's length in k-blocks), and the cuts
// are the greedy ones under the smallest per-cluster charge that covers the
// range: every piece takes as many units as the charge allows, ending at
// the tile boundary instead when the short ending would cost more.
bool stream_k_feasible(long long units, int num_kb, int clusters, int dp_tiles, long long e_kb, long long limit,
                       unsigned int *cuts) {
    long long x = 0;
    cuts[0] = 0;
    for (int c = 0; c < clusters; ++c) {
        long long y = x + limit < units ? x + limit : units;
        const long long b = y % num_kb, ts = y - b;
        const bool dp_follows = c < dp_tiles;
        if (b > 0 && b < e_kb && ts > x && dp_follows && (ts - x) + e_kb > limit) y = ts;
        cuts[c + 1] = static_cast<unsigned int>(y);
        x = y;
    }
    return x == units;
}

void stream_k_cuts(long long units, int num_kb, int clusters, int dp_tiles, long long e_kb, unsigned int *cuts) {
    long long lo = (units + clusters - 1) / clusters, hi = lo + e_kb;  // hi always covers the range
    while (lo < hi) {
        const long long mid = (lo + hi) / 2;
        if (stream_k_feasible(units, num_kb, clusters, dp_tiles, e_kb, mid, cuts))
            hi = mid;
        else
            lo = mid + 1;
    }
    stream_k_feasible(units, num_kb, clusters, dp_tiles, e_kb, lo, cuts);
}

void choose_schedule(int64_t tiles, int num_kb, int max_clusters, bool have_ws, int mode, int bn, int *dp_tiles,
                     long long *sk_units, unsigned int *cuts, int *clusters) {
    *dp_tiles = static_cast<int>(tiles);
    *sk_units = 0;
    *clusters = static_cast<int>(tiles < max_clusters ? tiles : max_clusters);
    if (!have_ws || mode == GEMM_SCHED_TILES || max_clusters <= 0 || max_clusters > kMaxSkClusters) return;
    int64_t dp = 0;
    if (mode != GEMM_SCHED_STREAM_K) {
        if (tiles % max_clusters == 0) return;
        const int64_t waves = tiles / max_clusters;
        const double idle = 1.0 - static_cast<double>(tiles) / static_cast<double>((waves + 1) * max_clusters);
        if (waves < 2 || num_kb < 48 || idle < 0.10) return;
        dp = (waves - 1) * max_clusters;
    }
    const long long units = static_cast<long long>(tiles - dp) * num_kb;
    if (units < 8LL * max_clusters || units > 0xFFFFFFFFLL) return;
    *dp_tiles = static_cast<int>(dp);
    *sk_units = units;
    *clusters = max_clusters;
    // An epilogue lasts about as long as 16 k-blocks of a 256-wide tile's MMAs
    // (fewer columns per k-block make each k-block proportionally shorter).
    const long long e_kb = 16LL * 256 / (bn > 0 ? bn : 256);
    stream_k_cuts(units, num_kb, max_clusters, static_cast<int>(dp), e_kb, cuts);
}

int pair_max_clusters_for(int ab, int cd, int cl) {
    switch (ab) {
    case GEMM_F16: return pair_max_clusters_f16(cd, cl);
    case GEMM_BF16: return pair_max_clusters_bf16(cd, cl);
    case GEMM_E4M3: return pair_max_clusters_e4m3(cd, cl);
    case kDtTF32x3: return cl == 2 ? pair_max_clusters_tf32x3(cd) : 0;
    default: return 0;
    }
}

// Resident clusters of `cl` (2 or 4) CTAs of the pair kernel on this device (cached).
int device_max_clusters(DeviceState *d, int ab, int cd, int cl = 2) {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    int &v = d->max_clusters[cl == 4 ? 1 : 0][ab][cd];
    if (v < 0) v = pair_max_clusters_for(ab, cd, cl);
    return v;
}

// Clusters of two pairs (A shared by multicast) or of one pair.  Two pairs
// need the A tile to split into whole TMA boxes between them (always for a
// K-contiguous A; for an M-contiguous A only with 16-bit elements, two
// 128-byte boxes per 128 rows), and AUTO wants the tile columns to pair up
// evenly, so no pair computes a tile outside the matrix.  Four-CTA clusters
// may fit on fewer SMs than pairs do (GB300: 36 clusters = 144 SMs against
// 76 pairs = 152).  Measured there, multicast lowers a launch's fixed cost
// (about 24 -> 20 us at 4096^3) and raises the per-SM rate by about 3%, so it
// wins while the fixed cost weighs (fp16 4096^3 +2.7%, bf16 M=2048 N=K=4096
// +1%: up to about 4 waves of pair tiles) and loses once the lost SMs do
// (bf16 8192^3 -1.4%, M=8192 N=K=4096 -4%).  AUTO follows that: two-pair
// clusters when they lose no SM, or when there are at most 4 waves of tiles.
int choose_cluster(int64_t tiles, int64_t tiles_n, int max_pairs, int max_quads, bool a_splits, int mode) {
    if (mode == GEMM_MCAST_OFF || !a_splits || max_quads <= 0) return 2;
    if (mode == GEMM_MCAST_ON) return 4;
    if (tiles_n % 2 != 0) return 2;
    return (2 * max_quads >= max_pairs || tiles <= 4LL * max_pairs) ? 4 : 2;
}

struct TileChoice {
    int kind = 1;  // 1: one SM per 128 x bn tile; 2: a pair of SMs per 256 x bn tile
    int bn = 256;
};

// Cost model.  Every SM computes 128 rows x bn columns per tile, so a tile
// takes time ~ bn / eff, where eff is the tensor-pipe duty cycle that shared
// memory bandwidth (~128 B/clk/SM) allows: per 16-deep k slice the MMA reads
// A (4 KB) and its B columns and TMA writes the same bytes.
//   one SM, 128 x bn:  (4096 + 32 bn) * 2 bytes per bn/2 clk
//   pair, 256 x bn:    (4096 + 16 bn) * 2 bytes per bn/2 clk
// Time = ceil(tiles / concurrent tiles) * bn / eff: wave quantisation over the
// SMs (one-SM) or the resident clusters (pair) is the other term.  Pair widths
// between 128 and 256 are not candidates: measured on GB300 they lose more
// per tile (e.g. fp8 4096^3: 2314 TFLOP/s at 224 vs 2684 at 256) than wave
// balance gains; they stay reachable through the tile policy.
TileChoice choose_tile(int64_t M, int64_t N, int num_sms, int max_clusters, int policy, int policy_bn) {
    auto cdiv = [](int64_t a, int64_t b) { return (a + b - 1) / b; };
    auto eff_of = [](int kind, int bn) {
        const double bytes_per_clk = kind == 2 ? 4.0 * (4096.0 + 16.0 * bn) / bn : 4.0 * (4096.0 + 32.0 * bn) / bn;
        return bytes_per_clk <= 128.0 ? 1.0 : 128.0 / bytes_per_clk;
    };
    TileChoice best;
    double best_t = 1e300;
    auto consider = [&](int kind, int bn) {
        int64_t tiles, units;
        if (kind == 2) {
            if (max_clusters <= 0) return;
            tiles = cdiv(M, 256) * cdiv(N, bn);
            units = max_clusters;
        } else {
            tiles = cdiv(M, 128) * cdiv(N, bn);
            units = num_sms;
        }
        const double t = static_cast<double>(cdiv(tiles, units)) * bn / eff_of(kind, bn);
        if (t < best_t * (1.0 - 1e-9)) {
            best_t = t;
            best.kind = kind;
            best.bn = bn;
        }
    };
    static const int pair_widths[] = {256, 128};
    if (policy == GEMM_TILE_1SM_256) return TileChoice{1, 256};
    if (policy == GEMM_TILE_1SM_128) return TileChoice{1, 128};
    if (policy == GEMM_TILE_PAIR && max_clusters > 0) {
        if (policy_bn > 0) return TileChoice{2, policy_bn};
        for (int bn : pair_widths) consider(2, bn);
        return best;
    }
    for (int bn : pair_widths) consider(2, bn);
    consider(1, 256);
    consider(1, 128);
    return best;
}

cudaError_t launch_pair(int ab, int cd, int cl, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                        const TcArgs &args, int clusters, cudaStream_t s) {
    switch (ab) {
    case GEMM_F16: return launch_pair_f16(cd, cl, ta, tb, tc, args, clusters, s);
    case GEMM_BF16: return launch_pair_bf16(cd, cl, ta, tb, tc, args, clusters, s);
    case GEMM_E4M3: return launch_pair_e4m3(cd, cl, ta, tb, tc, args, clusters, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tc(int ab, int cd, int bn, const CUtensorMap &ta, const CUtensorMap &tb, const TcArgs &args,
                      int grid, cudaStream_t s) {
    switch (ab) {
    case GEMM_F16: return launch_tcgen05_f16(cd, bn, ta, tb, args, grid, s);
    case GEMM_BF16: return launch_tcgen05_bf16(cd, bn, ta, tb, args, grid, s);
    case GEMM_E4M3: return launch_tcgen05_e4m3(cd, bn, ta, tb, args, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

EpiParams make_epi(int64_t M, int64_t N, void *C, int64_t ldc, int cd, float alpha, float beta, const float *bias,
                   int epi) {
    EpiParams e = {};  // every field defined, including those later calls fill in
    e.M = static_cast<int>(M);
    e.N = static_cast<int>(N);
    e.C = C;
    e.ldc = ldc;
    e.bias = bias;
    e.alpha = alpha;
    e.beta = beta;
    e.epilogue = epi;
    const bool c_al = (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && (ldc * elem_bytes(cd)) % 16 == 0;
    const bool b_al = epi == GEMM_EPI_NONE || (reinterpret_cast<uintptr_t>(bias) & 15u) == 0;
    e.c_vec = (c_al && b_al) ? 1 : 0;
    e.c_tma = 0;  // set by the pair-kernel launch once C's tensor map is encoded
    e.swap = 0;   // set by the pair-kernel launch when it computes C^T = B^T A^T
    e.scaled = 0;  // scales, fp8 output scale and amax: set by gemm_ex
    e.alpha_scale = e.row_scale = e.col_scale = nullptr;
    e.out_scale = nullptr;
    e.amax = nullptr;
    e.residual = nullptr;  // residual: set by gemm_ex
    e.ldr = 0;
    e.r_vec = 0;
    return e;
}

// fp32 GEMM as 3xTF32: split A and B into the workspace, then the pair kernel
// on the stacked hi/lo arrays (whole tiles, 256 x 256).
gemm_status_t gemm_tf32x3(int64_t M, int64_t N, int64_t K, const void *A, int64_t sam, int64_t sak, const void *B,
                          int64_t sbk, int64_t sbn, const EpiParams &e, void *workspace, int max_clusters,
                          DeviceState *dev, cudaStream_t s, gemm_launch_info_t *info, bool direct_c) {
    const int64_t pitch = tf32x3_pitch(K);
    float *a2 = static_cast<float *>(workspace);
    float *b2 = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                          round256(2 * static_cast<size_t>(M) * pitch * 4));
    if (launch_tf32_split(static_cast<const float *>(A), M, K, sam, sak, a2, pitch, s) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (launch_tf32_split(static_cast<const float *>(B), N, K, sbn, sbk, b2, pitch, s) != cudaSuccess)
        return GEMM_ERR_CUDA;
    const int bn = 256;
    CUtensorMap ta, tb;
    gemm_status_t st;
    if ((st = encode_2d_dt(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a2, K, 2 * M, pitch, 32, 128)) != GEMM_OK)
        return st;
    if ((st = encode_2d_dt(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, b2, K, 2 * N, pitch, 32, bn / 2)) != GEMM_OK)
        return st;
    TcArgs t = {};
    t.e = e;
    t.K = static_cast<int>(K);
    t.tiles_m = static_cast<int>((M + 255) / 256);
    t.tiles_n = static_cast<int>((N + bn - 1) / bn);
    t.num_tiles = t.tiles_m * t.tiles_n;
    t.num_kb = static_cast<int>((K + 31) / 32);
    t.group_m = 8;
    t.a_mn_major = 0;
    t.b_mn_major = 0;
    t.status = dev->status;
    t.bn = bn;
    t.stage_tx = 2u * (128u * 128u + static_cast<uint32_t>(bn / 2) * 128u);
    t.dp_tiles = t.num_tiles;
    t.sk_units = 0;
    std::fill(std::begin(t.sk_cut), std::end(t.sk_cut), 0u);
    t.partial = nullptr;
    t.flags = nullptr;
    t.epoch = 0;
    t.lo_row_a = static_cast<int>(M);
    t.lo_row_b = static_cast<int>(N);
    CUtensorMap tc;
    std::memset(&tc, 0, sizeof(tc));
    t.e.c_tma = (!direct_c && encode_c(&tc, GEMM_F32, e.C, M, N, e.ldc)) ? 1 : 0;
    const int clusters = t.num_tiles < max_clusters ? t.num_tiles : max_clusters;
    info->path = GEMM_PATH_TCGEN05;
    info->kind = 2;
    info->bn = bn;
    info->cluster_ctas = 2;
    info->grid_ctas = 2 * clusters;
    info->tiles = t.num_tiles;
    info->tf32x3 = 1;
    return launch_pair_tf32x3(GEMM_F32, ta, tb, tc, t, clusters, s) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

extern "C" {

gemm_status_t gemm_query_path(int64_t M, int64_t N, int64_t K, gemm_dtype_t ab_dtype, const void *A,
                              int64_t a_stride_m, int64_t a_stride_k, const void *B, int64_t b_stride_k,
                              int64_t b_stride_n, const void *C, int64_t ldc, gemm_dtype_t c_dtype, float alpha,
                              float beta, const float *bias, gemm_epilogue_t epilogue, gemm_path_t *path) {
    (void)beta;
    if (path == nullptr) return GEMM_ERR_INVALID_ARG;
    Plan plan;
    gemm_status_t st = make_plan(M, N, K, ab_dtype, A, a_stride_m, a_stride_k, B, b_stride_k, b_stride_n, C, ldc,
                                 c_dtype, alpha, bias, epilogue, &plan);
    if (st == GEMM_OK) *path = plan.path;
    return st;
}

size_t gemm_workspace_size(int64_t M, int64_t N, int64_t K, gemm_dtype_t ab_dtype) {
    if (ab_dtype == GEMM_F32) return tf32x3_workspace_bytes(M, N, K);
    if (ab_dtype != GEMM_F16 && ab_dtype != GEMM_BF16 && ab_dtype != GEMM_E4M3) return 0;
    DeviceState *dev = nullptr;
    if (device_state(&dev) != GEMM_OK) {
        cudaGetLastError();
        return 0;
    }
    return workspace_bytes_for(dev->num_sms / 2);
}

gemm_status_t gemm_set_schedule(gemm_schedule_t schedule) {
    if (schedule < GEMM_SCHED_AUTO || schedule > GEMM_SCHED_STREAM_K) return GEMM_ERR_INVALID_ARG;
    t_tuning.schedule = schedule;
    return GEMM_OK;
}

gemm_status_t gemm_ex(int64_t M, int64_t N, int64_t K, gemm_dtype_t ab_dtype, const void *A, int64_t a_stride_m,
                      int64_t a_stride_k, const void *B, int64_t b_stride_k, int64_t b_stride_n, void *C, int64_t ldc,
                      gemm_dtype_t c_dtype, float alpha, float beta, const float *bias, gemm_epilogue_t epilogue,
                      const gemm_scales_t *scales, void *workspace, size_t workspace_bytes, gemm_stream_t stream) {
    // E4M3 outputs: through gemm_ex only, written (beta == 0), from 16-bit or fp8 inputs.
    if (c_dtype == GEMM_E4M3 && (beta != 0.0f || ab_dtype == GEMM_F32)) return GEMM_ERR_UNSUPPORTED;
    Plan plan;
    gemm_status_t st = make_plan(M, N, K, ab_dtype, A, a_stride_m, a_stride_k, B, b_stride_k, b_stride_n, C, ldc,
                                 c_dtype, alpha, bias, epilogue, &plan, /*fp8_out=*/true);
    gemm_launch_info_t info = {};
    info.path = plan.path;
    if (st != GEMM_OK || plan.path == GEMM_PATH_NOOP) return record(st, info);
    if (!driver_fns().ok) return GEMM_ERR_CUDA;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != GEMM_OK) return st;

    const int es = elem_bytes(ab_dtype), ces = elem_bytes(c_dtype);
    if ((st = check_range(C, span_bytes(M, N, ldc, 1, ces))) != GEMM_OK) return st;
    if (epilogue != GEMM_EPI_NONE && (st = check_range(bias, static_cast<size_t>(N) * 4)) != GEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    EpiParams e = make_epi(M, N, C, ldc, c_dtype, alpha, beta, bias, epilogue);
    if (scales != nullptr && plan.path != GEMM_PATH_EPILOGUE_ONLY) {
        if (scales->alpha_scale && (st = check_range(scales->alpha_scale, 4)) != GEMM_OK) return st;
        if (scales->row_scale && (st = check_range(scales->row_scale, static_cast<size_t>(M) * 4)) != GEMM_OK)
            return st;
        if (scales->col_scale && (st = check_range(scales->col_scale, static_cast<size_t>(N) * 4)) != GEMM_OK)
            return st;
        e.alpha_scale = scales->alpha_scale;
        e.row_scale = scales->row_scale;
        e.col_scale = scales->col_scale;
    }
    if (scales != nullptr) {
        if (scales->out_scale && (st = check_range(scales->out_scale, 4)) != GEMM_OK) return st;
        if (scales->amax && (st = check_range(scales->amax, 4)) != GEMM_OK) return st;
        e.out_scale = c_dtype == GEMM_E4M3 ? scales->out_scale : nullptr;
        e.amax = scales->amax;
        if (scales->residual != nullptr) {
            // post-activation residual, M x ldr in the output type (not with an E4M3 output)
            if (c_dtype == GEMM_E4M3) return GEMM_ERR_UNSUPPORTED;
            if (scales->ldr < N) return GEMM_ERR_INVALID_ARG;
            if ((st = check_range(scales->residual, span_bytes(M, N, scales->ldr, 1, ces))) != GEMM_OK) return st;
            e.residual = scales->residual;
            e.ldr = scales->ldr;
            e.r_vec = ((reinterpret_cast<uintptr_t>(scales->residual) & 15u) == 0 && (scales->ldr * ces) % 16 == 0)
                          ? 1 : 0;
        }
    }
    e.scaled = (e.alpha_scale || e.row_scale || e.col_scale || e.out_scale || e.amax || e.residual ||
                c_dtype == GEMM_E4M3) ? 1 : 0;
    // E4M3 outputs and the amax reduction use the direct stores (no staged C).
    const bool direct_c = c_dtype == GEMM_E4M3 || e.amax != nullptr;

    if (plan.path == GEMM_PATH_EPILOGUE_ONLY)
        return record(launch_epilogue_only(c_dtype, e, s) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA, info);

    bool a_local = false, b_local = false;  // device memory of this device (multicast needs it)
    if ((st = check_range(A, span_bytes(M, K, a_stride_m, a_stride_k, es), dev->ordinal, &a_local)) != GEMM_OK)
        return st;
    if ((st = check_range(B, span_bytes(K, N, b_stride_k, b_stride_n, es), dev->ordinal, &b_local)) != GEMM_OK)
        return st;

    if (plan.path == GEMM_PATH_SIMT && ab_dtype == GEMM_F32) {
        // fp32 inputs: 3xTF32 on the tensor cores when the caller's workspace
        // holds the split operands; otherwise the FFMA kernel below.
        const size_t need = tf32x3_workspace_bytes(M, N, K);
        const int max_clusters = device_max_clusters(dev, kDtTF32x3, GEMM_F32);
        if (need > 0 && workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0 &&
            workspace_bytes >= need && max_clusters > 0) {
            if ((st = check_range(workspace, need)) != GEMM_OK) return st;
            return record(gemm_tf32x3(M, N, K, A, a_stride_m, a_stride_k, B, b_stride_k, b_stride_n, e, workspace,
                                      max_clusters, dev, s, &info, direct_c),
                          info);
        }
    }
    if (plan.path == GEMM_PATH_SIMT) {
        SimtArgs a = {};
        a.e = e;
        a.K = static_cast<int>(K);
        a.A = A; a.sam = a_stride_m; a.sak = a_stride_k;
        a.B = B; a.sbk = b_stride_k; a.sbn = b_stride_n;
        return record(launch_simt(ab_dtype, c_dtype, a, s) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA, info);
    }

    // tcgen05 path: one SM or a pair of SMs per tile, by the cost model.  The
    // pair kernel may run the transposed problem C^T = B^T A^T (kernel rows =
    // output columns), see gemm_operand_order_t.
    const int max_clusters = device_max_clusters(dev, ab_dtype, c_dtype);
    CUtensorMap tcm;
    std::memset(&tcm, 0, sizeof(tcm));
    const bool c_tma = !direct_c && encode_c(&tcm, c_dtype, C, M, N, ldc);
    const int order = t_tuning.operand_order;
    bool swap = c_tma && c_dtype != GEMM_F32 && order != GEMM_ORDER_AS_GIVEN &&
                (order == GEMM_ORDER_TRANSPOSED ||
                 (plan.b.mn_major && !plan.a.mn_major && ab_dtype != GEMM_E4M3));
    TileChoice tc;
    if (swap) {
        tc = choose_tile(N, M, dev->num_sms, max_clusters, t_tuning.tile_policy, t_tuning.tile_policy_bn);
        if (tc.kind != 2) swap = false;  // the one-SM kernel runs the problem as given
    }
    if (!swap) {
        // E4M3 outputs are built for the pair kernel only.
        const int policy = c_dtype == GEMM_E4M3 ? GEMM_TILE_PAIR : t_tuning.tile_policy;
        tc = choose_tile(M, N, dev->num_sms, max_clusters, policy, t_tuning.tile_policy_bn);
    }
    // The kernel's problem: Mk x Nk, first operand (Mk x K), second (Nk x K).
    const int64_t Mk = swap ? N : M, Nk = swap ? M : N;
    const Operand &op1 = swap ? plan.b : plan.a, &op2 = swap ? plan.a : plan.b;
    const int bk = 128 / es;
    const int64_t rows_per_tile = tc.kind == 2 ? 256 : 128;
    const int64_t tiles_m = (Mk + rows_per_tile - 1) / rows_per_tile;
    const int64_t tiles_n = (Nk + tc.bn - 1) / tc.bn;
    // The second operand's box covers this SM's columns: the whole tile (one SM) or half of it (pair).
    const uint32_t b_box = static_cast<uint32_t>(tc.kind == 2 ? tc.bn / 2 : tc.bn);
    // Pair kernel: clusters of one pair, or of two pairs that each fetch half
    // of a CTA's A rows (a 64-row box when A is K-contiguous) and multicast
    // them.  A multicast tensor map covers only this device's own memory: the
    // kernel's first operand must be a device allocation of the current
    // device, or the call runs one-pair clusters (no multicast).
    int cl = 2, max_quads = 0;
    if (tc.kind == 2) {
        const int mode = t_tuning.multicast;
        const bool a_splits = !op1.mn_major || es == 2;
        const bool op1_local = swap ? b_local : a_local;
        if (mode != GEMM_MCAST_OFF && a_splits && op1_local)
            max_quads = device_max_clusters(dev, ab_dtype, c_dtype, 4);
        cl = choose_cluster(tiles_m * tiles_n, tiles_n, max_clusters, max_quads, a_splits, mode);
    }
    const uint32_t a_box = cl == 4 ? 64u : 128u;
    CUtensorMap ta, tb;
    if (swap) {
        if ((st = encode_operand(&ta, ab_dtype, B, plan.b, N, K, b_stride_n, b_stride_k, a_box)) != GEMM_OK)
            return st;
        if ((st = encode_operand(&tb, ab_dtype, A, plan.a, M, K, a_stride_m, a_stride_k, b_box)) != GEMM_OK)
            return st;
    } else {
        if ((st = encode_operand(&ta, ab_dtype, A, plan.a, M, K, a_stride_m, a_stride_k, a_box)) != GEMM_OK)
            return st;
        if ((st = encode_operand(&tb, ab_dtype, B, plan.b, N, K, b_stride_n, b_stride_k, b_box)) != GEMM_OK)
            return st;
    }
    TcArgs t = {};
    t.e = e;
    t.K = static_cast<int>(K);
    t.tiles_m = static_cast<int>(tiles_m);
    t.tiles_n = static_cast<int>(tiles_n);
    t.num_tiles = static_cast<int>(tiles_m * tiles_n);
    t.num_kb = static_cast<int>((K + bk - 1) / bk);
    t.group_m = 8;
    t.a_mn_major = op1.mn_major ? 1u : 0u;
    t.b_mn_major = op2.mn_major ? 1u : 0u;
    t.status = dev->status;
    t.bn = tc.bn;
    const uint32_t swz = 128u / es;
    const uint32_t b_bytes = op2.mn_major ? ((b_box + swz - 1) / swz) * 128u * bk : b_box * 128u;
    t.stage_tx = 128u * 128u + b_bytes;
    t.dp_tiles = t.num_tiles;
    t.sk_units = 0;
    std::fill(std::begin(t.sk_cut), std::end(t.sk_cut), 0u);
    t.partial = nullptr;
    t.flags = nullptr;
    t.epoch = 0;
    cudaError_t err;
    if (tc.kind == 2) {
        // With two pairs per cluster the schedule's unit is a pair of tiles side
        // by side along N (the second one may lie outside the matrix when
        // forced with an odd number of tile columns).
        const int max_units = cl == 4 ? max_quads : max_clusters;
        const int slot_pairs = cl == 4 ? 2 * max_quads : max_clusters;  // partial-sum slots (per SM pair)
        if (cl == 4) {
            t.tiles_n = static_cast<int>((tiles_n + 1) / 2);
            t.num_tiles = t.tiles_m * t.tiles_n;
            t.dp_tiles = t.num_tiles;
        }
        const bool have_ws = workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0 &&
                             workspace_bytes >= workspace_bytes_for(slot_pairs);
        int clusters = 0;
        choose_schedule(t.num_tiles, t.num_kb, max_units, have_ws, t_tuning.schedule, t.bn, &t.dp_tiles,
                        &t.sk_units, t.sk_cut, &clusters);
        if (t.sk_units > 0) {
            if ((st = check_range(workspace, workspace_bytes_for(slot_pairs))) != GEMM_OK) return st;
            t.partial = static_cast<float *>(workspace);
            t.flags = reinterpret_cast<unsigned int *>(static_cast<char *>(workspace) + partial_bytes(slot_pairs));
            t.epoch = next_epoch();
        }
        t.e.c_tma = c_tma ? 1 : 0;
        t.e.swap = swap ? 1 : 0;
        info.kind = 2;
        info.transposed = swap ? 1 : 0;
        info.cluster_ctas = cl;
        info.grid_ctas = cl * clusters;
        info.stream_k_tiles = t.num_tiles - t.dp_tiles;
        err = launch_pair(ab_dtype, c_dtype, cl, ta, tb, tcm, t, clusters, s);
    } else {
        const int grid = static_cast<int>(t.num_tiles < dev->num_sms ? t.num_tiles : dev->num_sms);
        info.kind = 1;
        info.cluster_ctas = 1;
        info.grid_ctas = grid;
        err = launch_tc(ab_dtype, c_dtype, tc.bn, ta, tb, t, grid, s);
    }
    info.bn = tc.bn;
    info.tiles = t.num_tiles;
    return record(err == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA, info);
}

gemm_status_t gemm_last_launch(gemm_launch_info_t *info) {
    if (info == nullptr) return GEMM_ERR_INVALID_ARG;
    *info = t_last_launch;
    return GEMM_OK;
}

gemm_status_t gemm(int64_t M, int64_t N, int64_t K, gemm_dtype_t ab_dtype, const void *A, int64_t a_stride_m,
                   int64_t a_stride_k, const void *B, int64_t b_stride_k, int64_t b_stride_n, void *C, int64_t ldc,
                   gemm_dtype_t c_dtype, float alpha, float beta, const float *bias, gemm_epilogue_t epilogue,
                   void *workspace, size_t workspace_bytes, gemm_stream_t stream) {
    if (c_dtype == GEMM_E4M3) return GEMM_ERR_UNSUPPORTED;  // fp8 outputs: gemm_ex (with their scale and amax)
    return gemm_ex(M, N, K, ab_dtype, A, a_stride_m, a_stride_k, B, b_stride_k, b_stride_n, C, ldc, c_dtype, alpha,
                   beta, bias, epilogue, nullptr, workspace, workspace_bytes, stream);
}

gemm_status_t gemm_set_operand_order(gemm_operand_order_t order) {
    if (order < GEMM_ORDER_AUTO || order > GEMM_ORDER_TRANSPOSED) return GEMM_ERR_INVALID_ARG;
    t_tuning.operand_order = order;
    return GEMM_OK;
}

gemm_status_t gemm_set_multicast(gemm_multicast_t mode) {
    if (mode < GEMM_MCAST_AUTO || mode > GEMM_MCAST_ON) return GEMM_ERR_INVALID_ARG;
    t_tuning.multicast = mode;
    return GEMM_OK;
}

gemm_status_t gemm_set_tile_policy(gemm_tile_policy_t policy, int bn) {
    if (policy < GEMM_TILE_AUTO || policy > GEMM_TILE_PAIR) return GEMM_ERR_INVALID_ARG;
    if (bn != 0 && (policy != GEMM_TILE_PAIR || bn < 128 || bn > 256 || bn % 32 != 0)) return GEMM_ERR_INVALID_ARG;
    t_tuning.tile_policy_bn = bn;
    t_tuning.tile_policy = policy;
    return GEMM_OK;
}

gemm_status_t gemm_query_tile(int64_t M, int64_t N, int64_t K, gemm_dtype_t ab_dtype, gemm_dtype_t c_dtype,
                              int *kind, int *bn, int *units) {
    (void)K;
    if (kind == nullptr || bn == nullptr || units == nullptr || M < 0 || N < 0) return GEMM_ERR_INVALID_ARG;
    if (!valid_dtype(ab_dtype) || !valid_dtype(c_dtype) || ab_dtype == GEMM_F32 || c_dtype == GEMM_E4M3)
        return GEMM_ERR_UNSUPPORTED;
    DeviceState *dev = nullptr;
    gemm_status_t st = device_state(&dev);
    if (st != GEMM_OK) return st;
    const int max_clusters = device_max_clusters(dev, ab_dtype, c_dtype);
    const TileChoice tc = choose_tile(M, N, dev->num_sms, max_clusters, t_tuning.tile_policy,
                                      t_tuning.tile_policy_bn);
    *kind = tc.kind;
    *bn = tc.bn;
    *units = tc.kind == 2 ? max_clusters : dev->num_sms;
    return GEMM_OK;
}

gemm_status_t gemm_bias_gelu(int64_t M, int64_t N, void *C, int64_t ldc, gemm_dtype_t c_dtype, const float *bias,
                             gemm_stream_t stream) {
    if (M < 0 || N < 0 || M > INT32_MAX || N > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    if (!valid_dtype(c_dtype) || c_dtype == GEMM_E4M3) return GEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return GEMM_OK;
    if (C == nullptr || bias == nullptr || ldc < N) return GEMM_ERR_INVALID_ARG;
    if (!driver_fns().ok) return GEMM_ERR_CUDA;
    gemm_status_t st;
    if ((st = check_range(C, span_bytes(M, N, ldc, 1, elem_bytes(c_dtype)))) != GEMM_OK) return st;
    if ((st = check_range(bias, static_cast<size_t>(N) * 4)) != GEMM_OK) return st;
    EpiParams e = make_epi(M, N, C, ldc, c_dtype, 1.0f, 0.0f, bias, GEMM_EPI_BIAS_GELU);
    return launch_bias_gelu(c_dtype, e, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? GEMM_OK
                                                                                                : GEMM_ERR_CUDA;
}

gemm_status_t gemm_baseline(gemm_baseline_t kind, int64_t M, int64_t N, int64_t K, gemm_dtype_t ab_dtype,
                            const void *A, int64_t a_stride_m, int64_t a_stride_k, const void *B, int64_t b_stride_k,
                            int64_t b_stride_n, void *C, int64_t ldc, gemm_dtype_t c_dtype, float alpha, float beta,
                            const float *bias, gemm_epilogue_t epilogue, gemm_stream_t stream) {
    if (kind != GEMM_BASELINE_SIMT && kind != GEMM_BASELINE_MMA_SYNC) return GEMM_ERR_INVALID_ARG;
    Plan plan;
    gemm_status_t st = make_plan(M, N, K, ab_dtype, A, a_stride_m, a_stride_k, B, b_stride_k, b_stride_n, C, ldc,
                                 c_dtype, alpha, bias, epilogue, &plan);
    if (st != GEMM_OK || plan.path == GEMM_PATH_NOOP) return st;
    const bool mma = kind == GEMM_BASELINE_MMA_SYNC;
    if (mma && plan.path != GEMM_PATH_EPILOGUE_ONLY) {
        if (ab_dtype != GEMM_F16 && ab_dtype != GEMM_BF16) return GEMM_ERR_UNSUPPORTED;
        if (!plan.a.tma || !plan.b.tma) return GEMM_ERR_UNSUPPORTED;
        const int64_t a_extent = plan.a.mn_major ? M : K, b_extent = plan.b.mn_major ? N : K;
        if (a_extent % 8 != 0 || b_extent % 8 != 0) return GEMM_ERR_UNSUPPORTED;
    }
    if (!driver_fns().ok) return GEMM_ERR_CUDA;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != GEMM_OK) return st;
    const int es = elem_bytes(ab_dtype), ces = elem_bytes(c_dtype);
    if ((st = check_range(C, span_bytes(M, N, ldc, 1, ces))) != GEMM_OK) return st;
    if (epilogue != GEMM_EPI_NONE && (st = check_range(bias, static_cast<size_t>(N) * 4)) != GEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const EpiParams e = make_epi(M, N, C, ldc, c_dtype, alpha, beta, bias, epilogue);
    if (plan.path == GEMM_PATH_EPILOGUE_ONLY)
        return launch_epilogue_only(c_dtype, e, s) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    if ((st = check_range(A, span_bytes(M, K, a_stride_m, a_stride_k, es))) != GEMM_OK) return st;
    if ((st = check_range(B, span_bytes(K, N, b_stride_k, b_stride_n, es))) != GEMM_OK) return st;
    SimtArgs a = {};
    a.e = e;
    a.K = static_cast<int>(K);
    a.A = A; a.sam = a_stride_m; a.sak = a_stride_k;
    a.B = B; a.sbk = b_stride_k; a.sbn = b_stride_n;
    const cudaError_t err = mma ? launch_mma_sync(ab_dtype, c_dtype, a, !plan.a.mn_major, !plan.b.mn_major, s)
                                : launch_simt(ab_dtype, c_dtype, a, s);
    return err == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// AUTO's choice of decode kernel for M rows of x, from 1 x / 8 x 16384 x 16384 on
// GB300: one row is HBM-streaming FFMA work (3.07 TB/s against 2.09 for the
// tensor-core kernel, whose integer unpacking then bounds it); from two rows
// on, the FFMA kernel re-reads x for every pair of weight rows (0.40 TB/s at
// eight rows) while the tensor-core kernel stays near 2 TB/s.
bool q4_auto_mma(int64_t M) { return M >= 2; }

gemm_status_t gemm_set_q4_kernel(gemm_q4_kernel_t kind) {
    if (kind < GEMM_Q4_AUTO || kind > GEMM_Q4_MMA) return GEMM_ERR_INVALID_ARG;
    t_tuning.q4_kernel = kind;
    return GEMM_OK;
}

gemm_status_t gemm_get_tuning(gemm_tuning_t *out) {
    if (out == nullptr) return GEMM_ERR_INVALID_ARG;
    out->tile_policy = t_tuning.tile_policy;
    out->tile_bn = t_tuning.tile_policy_bn;
    out->schedule = t_tuning.schedule;
    out->operand_order = t_tuning.operand_order;
    out->multicast = t_tuning.multicast;
    out->q4_kernel = t_tuning.q4_kernel;
    return GEMM_OK;
}

gemm_status_t gemm_q4(int64_t M, int64_t N, int64_t K, gemm_dtype_t x_dtype, const void *X, int64_t ldx,
                      const uint32_t *Wq, const void *scale_bias, void *C, int64_t ldc, gemm_dtype_t c_dtype,
                      float alpha, float beta, const float *bias, gemm_epilogue_t epilogue, gemm_stream_t stream) {
    if (M < 0 || N < 0 || K < 0 || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    if (!valid_dtype(x_dtype) || !valid_dtype(c_dtype)) return GEMM_ERR_INVALID_ARG;
    if (epilogue < GEMM_EPI_NONE || epilogue > GEMM_EPI_BIAS_RELU) return GEMM_ERR_INVALID_ARG;
    if (x_dtype != GEMM_F16 && x_dtype != GEMM_BF16) return GEMM_ERR_UNSUPPORTED;
    if (c_dtype == GEMM_E4M3) return GEMM_ERR_UNSUPPORTED;
    if (K % 64 != 0) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (M > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
    if (C == nullptr || ldc < N) return GEMM_ERR_INVALID_ARG;
    if (epilogue != GEMM_EPI_NONE && bias == nullptr) return GEMM_ERR_INVALID_ARG;
    const bool reads_x = K > 0 && alpha != 0.0f;
    if (reads_x) {
        if (X == nullptr || Wq == nullptr || scale_bias == nullptr || ldx < K) return GEMM_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(X) & 15u) != 0 || (ldx * 2) % 16 != 0 ||
            (reinterpret_cast<uintptr_t>(Wq) & 15u) != 0 || (reinterpret_cast<uintptr_t>(scale_bias) & 3u) != 0)
            return GEMM_ERR_MISALIGNED;
    }
    if (!driver_fns().ok) return GEMM_ERR_CUDA;
    DeviceState *dev = nullptr;
    gemm_status_t st;
    if ((st = device_state(&dev)) != GEMM_OK) return st;
    if ((st = check_range(C, span_bytes(M, N, ldc, 1, elem_bytes(c_dtype)))) != GEMM_OK) return st;
    if (epilogue != GEMM_EPI_NONE && (st = check_range(bias, static_cast<size_t>(N) * 4)) != GEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const EpiParams e = make_epi(M, N, C, ldc, c_dtype, alpha, beta, bias, epilogue);
    if (!reads_x) return launch_epilogue_only(c_dtype, e, s) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    if ((st = check_range(X, span_bytes(M, K, ldx, 1, 2))) != GEMM_OK) return st;
    if ((st = check_range(Wq, static_cast<size_t>(N) * static_cast<size_t>(K / 8) * 4)) != GEMM_OK) return st;
    if ((st = check_range(scale_bias, static_cast<size_t>(N) * static_cast<size_t>(K / 64) * 4)) != GEMM_OK)
        return st;
    Q4Args a = {};
    a.e = e;
    a.K = static_cast<int>(K);
    a.X = X;
    a.ldx = ldx;
    a.Wq = Wq;
    a.SB = static_cast<const uint32_t *>(scale_bias);
    a.status = dev->status;
    if (M > kQ4MaxRows) {
        // Prefill: the tensor-core product with W dequantised into tensor memory.
        CUtensorMap tmX, tmW;
        if ((st = encode_2d(&tmX, x_dtype, X, K, M, ldx, 64, 128)) != GEMM_OK) return st;
        cuuint64_t wdims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
        cuuint64_t wstrides[1] = {static_cast<cuuint64_t>(K / 2)};
        cuuint32_t wbox[2] = {32u, 128u};
        cuuint32_t westr[2] = {1, 1};
        if (driver_fns().encode(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t *>(Wq), wdims, wstrides,
                                wbox, westr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return GEMM_ERR_CUDA;
        const long long tiles = ((N + 127) / 128) * ((M + 127) / 128);
        const int grid = static_cast<int>(tiles < dev->num_sms ? tiles : dev->num_sms);
        gemm_launch_info_t info = {};
        info.path = GEMM_PATH_TCGEN05;
        info.kind = 1;
        info.bn = 128;
        info.transposed = 1;
        info.cluster_ctas = 1;
        info.grid_ctas = grid;
        info.tiles = static_cast<int>(tiles);
        return record(launch_q4_prefill(x_dtype, c_dtype, tmX, tmW, a, grid, s) == cudaSuccess ? GEMM_OK
                                                                                                : GEMM_ERR_CUDA,
                      info);
    }
    const int kind = t_tuning.q4_kernel;
    if (!(kind == GEMM_Q4_MMA || (kind == GEMM_Q4_AUTO && q4_auto_mma(M))))
        return launch_q4_gemv(x_dtype, c_dtype, nullptr, a, s) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    // The tensor-core kernel's weight boxes: 32 rows x min(160, K/2) bytes of codes.
    a.w_pitch = static_cast<int>(K / 2 < 160 ? K / 2 : 160);
    CUtensorMap tmW;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(a.w_pitch), 32u};
    cuuint32_t estr[2] = {1, 1};
    if (driver_fns().encode(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t *>(Wq), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return GEMM_ERR_CUDA;
    return launch_q4_gemv(x_dtype, c_dtype, &tmW, a, s) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

size_t gemm_q4_workspace_size(int64_t M, int64_t N, int64_t K, gemm_dtype_t x_dtype) {
    if (M < GEMM_Q4_DEQUANT_ROWS || N <= 0 || K <= 0 || K % 64 != 0) return 0;
    if (x_dtype != GEMM_F16 && x_dtype != GEMM_BF16) return 0;
    return round256(static_cast<size_t>(N) * static_cast<size_t>(K) * 2) + gemm_workspace_size(M, N, K, x_dtype);
}

gemm_status_t gemm_q4_ws(int64_t M, int64_t N, int64_t K, gemm_dtype_t x_dtype, const void *X, int64_t ldx,
                         const uint32_t *Wq, const void *scale_bias, void *C, int64_t ldc, gemm_dtype_t c_dtype,
                         float alpha, float beta, const float *bias, gemm_epilogue_t epilogue, void *workspace,
                         size_t workspace_bytes, gemm_stream_t stream) {
    const size_t need = gemm_q4_workspace_size(M, N, K, x_dtype);
    const bool use = need > 0 && workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0 &&
                     workspace_bytes >= need && alpha != 0.0f;
    if (!use)
        return gemm_q4(M, N, K, x_dtype, X, ldx, Wq, scale_bias, C, ldc, c_dtype, alpha, beta, bias, epilogue,
                       stream);
    // gemm_q4's argument rules first (the dense path accepts more), then the two calls.
    if (N > INT32_MAX || K > INT32_MAX || M > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
    if (!valid_dtype(c_dtype)) return GEMM_ERR_INVALID_ARG;
    if (epilogue < GEMM_EPI_NONE || epilogue > GEMM_EPI_BIAS_RELU) return GEMM_ERR_INVALID_ARG;
    if (c_dtype == GEMM_E4M3) return GEMM_ERR_UNSUPPORTED;
    if (C == nullptr || ldc < N) return GEMM_ERR_INVALID_ARG;
    if (epilogue != GEMM_EPI_NONE && bias == nullptr) return GEMM_ERR_INVALID_ARG;
    if (X == nullptr || Wq == nullptr || scale_bias == nullptr || ldx < K) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(X) & 15u) != 0 || (ldx * 2) % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(Wq) & 15u) != 0 || (reinterpret_cast<uintptr_t>(scale_bias) & 3u) != 0)
        return GEMM_ERR_MISALIGNED;
    gemm_status_t st;
    if ((st = check_range(workspace, need)) != GEMM_OK) return st;
    unsigned char *W = static_cast<unsigned char *>(workspace);
    const size_t w_bytes = round256(static_cast<size_t>(N) * static_cast<size_t>(K) * 2);
    if ((st = gemm_q4_dequantize(N, K, Wq, scale_bias, W, x_dtype, stream)) != GEMM_OK) return st;
    // W is N x K row-major: as B (K x N) it is K-contiguous, b_stride_k = 1, b_stride_n = K.
    return gemm(M, N, K, x_dtype, X, ldx, 1, W, 1, K, C, ldc, c_dtype, alpha, beta, bias, epilogue, W + w_bytes,
                workspace_bytes - w_bytes, stream);
}

gemm_status_t gemm_q4_dequantize(int64_t N, int64_t K, const uint32_t *Wq, const void *scale_bias, void *W,
                                 gemm_dtype_t w_dtype, gemm_stream_t stream) {
    if (N < 0 || K < 0 || K % 64 != 0) return GEMM_ERR_INVALID_ARG;
    if (w_dtype != GEMM_F16 && w_dtype != GEMM_BF16) return valid_dtype(w_dtype) ? GEMM_ERR_UNSUPPORTED
                                                                                 : GEMM_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return GEMM_OK;
    if (Wq == nullptr || scale_bias == nullptr || W == nullptr) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(Wq) & 3u) != 0 || (reinterpret_cast<uintptr_t>(scale_bias) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(W) & 15u) != 0)
        return GEMM_ERR_MISALIGNED;
    if (!driver_fns().ok) return GEMM_ERR_CUDA;
    DeviceState *dev = nullptr;
    gemm_status_t st;
    if ((st = device_state(&dev)) != GEMM_OK) return st;
    if ((st = check_range(Wq, static_cast<size_t>(N) * static_cast<size_t>(K / 8) * 4)) != GEMM_OK) return st;
    if ((st = check_range(scale_bias, static_cast<size_t>(N) * static_cast<size_t>(K / 64) * 4)) != GEMM_OK)
        return st;
    if ((st = check_range(W, static_cast<size_t>(N) * static_cast<size_t>(K) * 2)) != GEMM_OK) return st;
    return launch_q4_dequantize(w_dtype, N, K, Wq, static_cast<const uint32_t *>(scale_bias), W,
                                reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GEMM_OK
               : GEMM_ERR_CUDA;
}

// ---------------------------------------------------------- block-scaled --

// Chunk columns of the packed scales: 4 blocks of 32 k per chunk, rounded up
// to whole stages (1 chunk for E4M3 elements, 2 for E2M1).
static int64_t mx_kc_count(int64_t K, int elem) {
    const int64_t per_stage = elem == GEMM_MX_E2M1 ? 2 : 1;
    const int64_t blocks = K / 32;
    return (blocks + 4 * per_stage - 1) / (4 * per_stage) * per_stage;
}

static size_t mx_pack_bytes(int64_t rows, int64_t K, int elem) {
    return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>(mx_kc_count(K, elem)) * 512;
}

size_t gemm_mx_workspace_size(int64_t M, int64_t N, int64_t K, gemm_mx_elem_t elem) {
    if (M <= 0 || N <= 0 || K <= 0 || K % 32 != 0 || (elem != GEMM_MX_E4M3 && elem != GEMM_MX_E2M1) ||
        M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return 0;
    return round256(mx_pack_bytes(M, K, elem)) + round256(mx_pack_bytes(N, K, elem));
}

gemm_status_t gemm_mx(int64_t M, int64_t N, int64_t K, gemm_mx_elem_t elem, const void *A, int64_t lda,
                      const uint8_t *a_scale, const void *B, int64_t ldb, const uint8_t *b_scale, void *C,
                      int64_t ldc, gemm_dtype_t c_dtype, float alpha, float beta, const float *bias,
                      gemm_epilogue_t epilogue, void *workspace, size_t workspace_bytes, gemm_stream_t stream) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (elem != GEMM_MX_E4M3 && elem != GEMM_MX_E2M1) return GEMM_ERR_INVALID_ARG;
    if (!valid_dtype(c_dtype)) return GEMM_ERR_INVALID_ARG;
    if (c_dtype == GEMM_E4M3) return GEMM_ERR_UNSUPPORTED;
    if (epilogue < GEMM_EPI_NONE || epilogue > GEMM_EPI_BIAS_RELU) return GEMM_ERR_INVALID_ARG;
    if (K % 32 != 0) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return record(GEMM_OK, gemm_launch_info_t{});
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
    if (C == nullptr || ldc < N) return GEMM_ERR_INVALID_ARG;
    if (epilogue != GEMM_EPI_NONE && bias == nullptr) return GEMM_ERR_INVALID_ARG;
    if (!driver_fns().ok) return GEMM_ERR_CUDA;
    DeviceState *dev = nullptr;
    gemm_status_t st;
    if ((st = device_state(&dev)) != GEMM_OK) return st;
    const int ces = elem_bytes(c_dtype);
    if ((st = check_range(C, span_bytes(M, N, ldc, 1, ces))) != GEMM_OK) return st;
    if (epilogue != GEMM_EPI_NONE && (st = check_range(bias, static_cast<size_t>(N) * 4)) != GEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const EpiParams e = make_epi(M, N, C, ldc, c_dtype, alpha, beta, bias, epilogue);
    gemm_launch_info_t info = {};
    if (K == 0 || alpha == 0.0f) {
        info.path = GEMM_PATH_EPILOGUE_ONLY;
        return record(launch_epilogue_only(c_dtype, e, s) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA, info);
    }
    if (A == nullptr || B == nullptr || a_scale == nullptr || b_scale == nullptr) return GEMM_ERR_INVALID_ARG;
    if (lda < K || ldb < K) return GEMM_ERR_INVALID_ARG;
    // Elements per byte, and the row pitches in bytes: whole bytes, TMA-able (16-byte multiples).
    const int64_t per_byte = elem == GEMM_MX_E2M1 ? 2 : 1;
    if (lda % per_byte != 0 || ldb % per_byte != 0) return GEMM_ERR_INVALID_ARG;
    const int64_t a_pitch = lda / per_byte, b_pitch = ldb / per_byte, k_bytes = K / per_byte;
    if ((reinterpret_cast<uintptr_t>(A) & 15u) != 0 || (reinterpret_cast<uintptr_t>(B) & 15u) != 0 ||
        (M > 1 && a_pitch % 16 != 0) || (N > 1 && b_pitch % 16 != 0))
        return GEMM_ERR_MISALIGNED;
    if ((st = check_range(A, static_cast<size_t>((M - 1) * a_pitch + k_bytes))) != GEMM_OK) return st;
    if ((st = check_range(B, static_cast<size_t>((N - 1) * b_pitch + k_bytes))) != GEMM_OK) return st;
    const int64_t blocks = K / 32;
    if ((st = check_range(a_scale, static_cast<size_t>(M * blocks))) != GEMM_OK) return st;
    if ((st = check_range(b_scale, static_cast<size_t>(N * blocks))) != GEMM_OK) return st;
    const size_t need = gemm_mx_workspace_size(M, N, K, elem);
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need)
        return GEMM_ERR_WORKSPACE;
    if ((st = check_range(workspace, need)) != GEMM_OK) return st;

    // Scales into the chunk layout the kernel copies to tensor memory.
    const int64_t kc = mx_kc_count(K, elem);
    unsigned char *sfa = static_cast<unsigned char *>(workspace);
    unsigned char *sfb = sfa + round256(mx_pack_bytes(M, K, elem));
    if (launch_mx_sf_pack(a_scale, M, blocks, sfa, (M + 127) / 128, kc, s) != cudaSuccess) return GEMM_ERR_CUDA;
    if (launch_mx_sf_pack(b_scale, N, blocks, sfb, (N + 127) / 128, kc, s) != cudaSuccess) return GEMM_ERR_CUDA;

    if (M > 128) {
        // SM pairs, 256 x 256 tiles (gemm_mx_pair.cu): operands as bytes in boxes of
        // 128 bytes of K x 128 rows (each CTA's half), 128-byte swizzle, zero fill; the
        // chunked scales as rows of 256 bytes, one box = one stage's chunks of a
        // 128-row block.  Up to 128 rows of A the one-SM kernel's 128 x 256 tiles
        // waste no half-empty pair tile.
        CUtensorMap ta, tb, tsa, tsb;
        if ((st = encode_2d(&ta, GEMM_E4M3, A, k_bytes, M, a_pitch, 128, 128)) != GEMM_OK) return st;
        if ((st = encode_2d(&tb, GEMM_E4M3, B, k_bytes, N, b_pitch, 128, 128)) != GEMM_OK) return st;
        const cuuint32_t sf_rows = static_cast<cuuint32_t>(elem == GEMM_MX_E2M1 ? 4 : 2);
        for (int o = 0; o < 2; ++o) {
            const int64_t rows = o == 0 ? M : N;
            cuuint64_t dims[2] = {256u, static_cast<cuuint64_t>(2 * ((rows + 127) / 128) * kc)};
            cuuint64_t strides[1] = {256u};
            cuuint32_t box[2] = {256u, sf_rows};
            cuuint32_t estr[2] = {1, 1};
            if (driver_fns().encode(o == 0 ? &tsa : &tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, o == 0 ? sfa : sfb, dims,
                                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return GEMM_ERR_CUDA;
        }
        MxArgs a = {};
        a.e = e;
        a.K = static_cast<int>(K);
        a.tiles_m = static_cast<int>((M + 255) / 256);
        a.tiles_n = static_cast<int>((N + 255) / 256);
        a.num_tiles = a.tiles_m * a.tiles_n;
        a.num_kb = static_cast<int>((k_bytes + 127) / 128);
        a.group_m = 8;
        a.sfa = sfa;
        a.sfb = sfb;
        a.kc_count = static_cast<int>(kc);
        a.status = dev->status;
        const int max_clusters = dev->num_sms / 2;
        const int clusters = a.num_tiles < max_clusters ? a.num_tiles : max_clusters;
        info.path = GEMM_PATH_TCGEN05;
        info.kind = 2;
        info.bn = 256;
        info.cluster_ctas = 2;
        info.grid_ctas = 2 * clusters;
        info.tiles = a.num_tiles;
        return record(launch_mx_pair(elem, c_dtype, ta, tb, tsa, tsb, a, clusters, s) == cudaSuccess ? GEMM_OK
                                                                                                      : GEMM_ERR_CUDA,
                      info);
    }

    // Operands as bytes: boxes of 128 bytes of K x 128 rows (A) or 256 rows (B), 128-byte
    // swizzle, zero fill.
    CUtensorMap ta, tb;
    if ((st = encode_2d(&ta, GEMM_E4M3, A, k_bytes, M, a_pitch, 128, 128)) != GEMM_OK) return st;
    if ((st = encode_2d(&tb, GEMM_E4M3, B, k_bytes, N, b_pitch, 128, 256)) != GEMM_OK) return st;
    MxArgs a = {};
    a.e = e;
    a.K = static_cast<int>(K);
    a.tiles_m = static_cast<int>((M + 127) / 128);
    a.tiles_n = static_cast<int>((N + 255) / 256);
    a.num_tiles = a.tiles_m * a.tiles_n;
    a.num_kb = static_cast<int>((k_bytes + 127) / 128);
    a.group_m = 8;
    a.sfa = sfa;
    a.sfb = sfb;
    a.kc_count = static_cast<int>(kc);
    a.status = dev->status;
    const int grid = a.num_tiles < dev->num_sms ? a.num_tiles : dev->num_sms;
    info.path = GEMM_PATH_TCGEN05;
    info.kind = 1;
    info.bn = 256;
    info.cluster_ctas = 1;
    info.grid_ctas = grid;
    info.tiles = a.num_tiles;
    return record(launch_mx(elem, c_dtype, ta, tb, a, grid, s) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA, info);
}

gemm_status_t gemm_wait_selftest(const unsigned int *never_set, uint64_t limit_ns, gemm_stream_t stream) {
    if (never_set == nullptr || limit_ns == 0 || limit_ns > 1000000000ull) return GEMM_ERR_INVALID_ARG;
    if (!driver_fns().ok) return GEMM_ERR_CUDA;
    DeviceState *dev = nullptr;
    gemm_status_t st = device_state(&dev);
    if (st != GEMM_OK) return st;
    if ((st = check_range(never_set, sizeof(unsigned int))) != GEMM_OK) return st;
    return launch_wait_selftest(never_set, limit_ns, dev->status, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? GEMM_OK
               : GEMM_ERR_CUDA;
}

gemm_status_t gemm_device_status(gemm_stream_t stream) {
    DeviceState *dev = nullptr;
    gemm_status_t st = device_state(&dev);
    if (st != GEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GEMM_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpyAsync(&word, dev->status, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (cudaMemsetAsync(dev->status, 0, sizeof(word), s) != cudaSuccess) return GEMM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GEMM_ERR_CUDA;
    return word != 0 ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

const char *gemm_status_string(gemm_status_t status) {
    switch (status) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_UNSUPPORTED: return "unsupported dtype combination or size";
    case GEMM_ERR_MISALIGNED: return "misaligned operand";
    case GEMM_ERR_WORKSPACE: return "workspace missing or too small";
    case GEMM_ERR_CUDA: return "CUDA runtime or driver call failed";
    case GEMM_ERR_TIMEOUT: return "a device-side wait timed out";
    default: return "unknown status";
    }
}

const char *gemm_version(void) { return "gemm_gb300 0.1 (sm_103a, tcgen05)"; }

}  // extern "C"
