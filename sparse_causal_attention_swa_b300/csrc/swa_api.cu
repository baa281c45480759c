// swa_api.cu -- the C ABI of libswa_b300.so: argument validation, TMA tensor maps, the
// strided tile list, and kernel launches.  Declarations and the contract of every entry
// point are in include/swa_b300.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>
#include <utility>
#include <vector>

#include "attn_fwd.cuh"
#include "attn_bwd.cuh"
#include "decode.cuh"
#include "swa_b300.h"

namespace {

using swa::BM;
using swa::BN;
using swa::KParams;

constexpr int kMaxDevices = 64;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per bounded wait

// Device status word: kernels record SWA_ERR_TIMEOUT here when a bounded wait runs out.
__device__ int g_status_word;

struct DeviceState {
    bool probed = false;
    bool supported = false;
    int* status = nullptr;  // device address of g_status_word
    int num_sms = 0;
    bool attr_set[2][3] = {};
    bool dec_attr_set[2][5] = {};
    bool bwd_attr_set[2][3] = {};
    // strided tile lists, keyed by (N, W, stride, rows per block, compact-key cap)
    std::map<std::tuple<int, int, int, int, int>, int*> tile_lists;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];

// The cause of the calling thread's last SWA_ERR_CUDA (read by swa_last_error_detail).
thread_local char t_err_detail[160] = "";

int cuda_fail(const char* what, const char* err) {
    std::snprintf(t_err_detail, sizeof(t_err_detail), "%s: %s", what, err ? err : "?");
    return SWA_ERR_CUDA;
}
int cuda_fail(const char* what, cudaError_t e) { return cuda_fail(what, cudaGetErrorName(e)); }
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return cuda_fail("cudaGetDevice", e0);
    if (dev < 0 || dev >= kMaxDevices) return SWA_ERR_UNSUPPORTED;
    // make the device's primary context current on this thread: the tensor-map encoder is a
    // driver call, and a thread that has made no runtime call yet (an autograd worker, say)
    // has no current context
    e0 = cudaSetDevice(dev);
    if (e0 != cudaSuccess) return cuda_fail("cudaSetDevice", e0);
    DeviceState& st = g_dev[dev];
    if (!st.probed) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return SWA_ERR_CUDA;
        st.supported = (major == 10 && minor == 3);
        if (st.supported) {
            if (cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess)
                return SWA_ERR_CUDA;
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return SWA_ERR_CUDA;
            st.status = static_cast<int*>(p);
        }
        st.probed = true;
    }
    if (!st.supported) return SWA_ERR_UNSUPPORTED;
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return SWA_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = &st;
    return SWA_OK;
}

// Process-lifetime cache of encoded tensor maps.  A map is a pure function of the values it
// encodes (base address, extents, strides, box), so a cached entry is bit for bit what a new
// encoding would produce and never goes stale: a buffer freed and re-allocated at the same
// address with the same shape is described by the same map.  A repeated call therefore
// encodes nothing.  Guarded by g_mutex (every caller of make_map holds it); bounded by
// dropping the whole cache when it reaches kMapCacheMax entries.
struct MapKey {
    uintptr_t base;
    long long rows, row_stride, nmat, mat_stride;
    int d, box_rows;
    bool operator<(const MapKey& o) const {
        return std::tie(base, rows, row_stride, nmat, mat_stride, d, box_rows) <
               std::tie(o.base, o.rows, o.row_stride, o.nmat, o.mat_stride, o.d, o.box_rows);
    }
};
constexpr size_t kMapCacheMax = 4096;
std::map<MapKey, CUtensorMap> g_map_cache;

// 3-D view [nmat][rows][d] of a bf16 tensor; consecutive rows are `row_stride` elements
// apart and consecutive matrices (heads) `mat_stride` elements apart.  The box is
// 64 columns (128 bytes, one swizzle span) x box_rows rows x 1 matrix, 128-byte swizzled.
int make_map(CUtensorMap* m, const void* base, int d, long long rows, long long row_stride,
             long long nmat, long long mat_stride, int box_rows = 128) {
    const MapKey key{reinterpret_cast<uintptr_t>(base), rows, row_stride, nmat, mat_stride, d,
                     box_rows};
    auto it = g_map_cache.find(key);
    if (it != g_map_cache.end()) {
        *m = it->second;
        return SWA_OK;
    }
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)nmat};
    cuuint64_t strides[2] = {(cuuint64_t)row_stride * 2, (cuuint64_t)mat_stride * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[64];
        std::snprintf(msg, sizeof(msg), "CUresult %d", (int)r);
        return cuda_fail("cuTensorMapEncodeTiled", msg);
    }
    if (g_map_cache.size() >= kMapCacheMax) g_map_cache.clear();
    g_map_cache.emplace(key, *m);
    return SWA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A plain launch whose error comes back from the launch call itself (never from the thread's
// last-error state, which may hold an earlier error of another library on the same thread).
template <typename... KArgs, typename... Args>
int launch_plain(void (*kern)(KArgs...), unsigned grid, unsigned block, cudaStream_t stream,
                 Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.stream = stream;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    return e == cudaSuccess ? SWA_OK : cuda_fail("cudaLaunchKernelEx", e);
}

int check_common(int B, int Hq, int Hkv, int N, int d, float scale) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1) return SWA_ERR_SHAPE;
    if (Hq % Hkv != 0) return SWA_ERR_SHAPE;
    // grid and TMA coordinate limits: rows and heads are 32-bit coordinates
    if ((long long)B * Hq > (1ll << 24) || (long long)N > (1ll << 30)) return SWA_ERR_SHAPE;
    if (d != 64 && d != 128) return SWA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale) || !(scale > 0.f)) return SWA_ERR_VALUE;
    return SWA_OK;
}

template <int D, int MODE>
int launch(const KParams& kp, int n_items, cudaStream_t stream, DeviceState& st) {
    using L = swa::SmemLayout<D, MODE>;
    auto kern = swa::attn_fwd_kernel<D, MODE>;
    bool& set = st.attr_set[D == 128 ? 1 : 0][MODE];
    if (!set) {
        const cudaError_t ea =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
        if (ea != cudaSuccess) return cuda_fail("cudaFuncSetAttribute (forward)", ea);
        set = true;
    }
    // persistent grid: one CTA per SM (tensor memory and shared memory allow no more),
    // each walking its share of the items
    KParams kq = kp;
    kq.n_items = n_items;
    const int grid = std::min(n_items, st.num_sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(swa::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::BYTES;
    cfg.stream = stream;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, kq);
    return e == cudaSuccess ? SWA_OK : cuda_fail("cudaLaunchKernelEx (forward)", e);
}

template <int MODE>
int dispatch(int d, const KParams& kp, int n_items, cudaStream_t stream, DeviceState& st) {
    if (d == 128) return launch<128, MODE>(kp, n_items, stream, st);
    return launch<64, MODE>(kp, n_items, stream, st);
}

void fill_common(KParams& kp, int B, int Hq, int Hkv, int N, int W, int stride, float scale,
                 void* out, DeviceState& st) {
    kp.out = static_cast<__nv_bfloat16*>(out);
    kp.tiles = nullptr;
    kp.status = st.status;
    kp.wait_limit_ns = kWaitLimitNs;
    kp.B = B;
    kp.Hq = Hq;
    kp.Hkv = Hkv;
    kp.N = N;
    kp.W = W;
    kp.stride = stride;
    kp.n_qtiles = (N + BM - 1) / BM;
    kp.scale_log2 = scale * 1.4426950408889634f;
    kp.scale = scale;
    kp.q_off = 0;
    kp.strided_cap = 0x7fffffff;
    kp.lambda = 0.f;
}

// Work items: two slots per CTA.  Query heads of one GQA group are paired when the group
// size is even; otherwise the slots are two consecutive row tiles of one head.
int n_items_for(const KParams& kp) {
    if (kp.pair_mode) return kp.B * kp.Hkv * ((kp.Hq / kp.Hkv) / 2) * kp.n_qtiles;
    return kp.B * kp.Hq * ((kp.n_qtiles + 1) / 2);
}

// The strided tile list: for every row block (the union of an item's rows), the compact
// strided-key tiles that hold keys 0, s, 2s, ... before the block's last window start,
// then the window tiles from the first row's window start to the block's last row.
int get_tile_list(DeviceState& st, int N, int W, int stride, int rows_per_block, int cap,
                  cudaStream_t stream, const int** out) {
    auto key = std::make_tuple(N, W, stride, rows_per_block, cap);
    auto it = st.tile_lists.find(key);
    if (it != st.tile_lists.end()) {
        *out = it->second;
        return SWA_OK;
    }
    const int nblk = (N + rows_per_block - 1) / rows_per_block;
    std::vector<int> offs(nblk + 1, 0), ents;
    for (int blk = 0; blk < nblk; ++blk) {
        const long long R0 = (long long)blk * rows_per_block;
        const long long R1 = std::min<long long>(R0 + rows_per_block, N) - 1;
        const long long lo0 = std::max<long long>(0, R0 - W + 1);
        const long long lo1 = std::max<long long>(0, R1 - W + 1);
        // multiples of s below lo1, at most cap of them
        const long long nkeys = std::min<long long>((lo1 + stride - 1) / stride, cap);
        const long long ncompact = (nkeys + BN - 1) / BN;
        for (long long c = 0; c < ncompact; ++c)
            ents.push_back((swa::TILE_KIND_STRIDED << swa::TILE_KIND_SHIFT) | (int)c);
        for (long long t = lo0 / BN; t <= R1 / BN; ++t)
            ents.push_back((swa::TILE_KIND_WINDOW << swa::TILE_KIND_SHIFT) | (int)t);
        offs[blk + 1] = (int)ents.size();
    }
    std::vector<int> host(offs);
    host.insert(host.end(), ents.begin(), ents.end());
    int* dptr = nullptr;
    if (cudaMalloc(&dptr, host.size() * sizeof(int)) != cudaSuccess) return SWA_ERR_CUDA;
    if (cudaMemcpyAsync(dptr, host.data(), host.size() * sizeof(int), cudaMemcpyHostToDevice,
                        stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaFree(dptr);
        return SWA_ERR_CUDA;
    }
    st.tile_lists[key] = dptr;
    *out = dptr;
    return SWA_OK;
}

// ---------------------------------------------------------------------------------------
// Allocation-free strided call: the tile list lives in one fixed device array.
// ---------------------------------------------------------------------------------------
static __device__ __align__(256) int g_noalloc_tiles[SWA_NOALLOC_TILE_CAPACITY];

struct NoAllocState {
    bool ready = false;
    int* tiles = nullptr;  // device address of g_noalloc_tiles on that device
};
NoAllocState g_noalloc[kMaxDevices];

__host__ __device__ inline void noalloc_block_counts(long long blk, int N, int W, int stride,
                                                     int rpb, long long* ncompact,
                                                     long long* wfirst, long long* wlast) {
    const long long R0 = blk * rpb;
    const long long R1 = (R0 + rpb < N ? R0 + rpb : N) - 1;
    const long long lo0 = R0 - W + 1 > 0 ? R0 - W + 1 : 0;
    const long long lo1 = R1 - W + 1 > 0 ? R1 - W + 1 : 0;
    const long long nkeys = (lo1 + stride - 1) / stride;
    *ncompact = (nkeys + BN - 1) / BN;
    *wfirst = lo0 / BN;
    *wlast = R1 / BN;
}

long long noalloc_list_length(int N, int W, int stride, int rpb) {
    const long long nblk = (N + rpb - 1) / rpb;
    long long len = nblk + 1;
    for (long long blk = 0; blk < nblk; ++blk) {
        long long nc, wf, wl;
        noalloc_block_counts(blk, N, W, stride, rpb, &nc, &wf, &wl);
        len += nc + (wl - wf + 1);
        if (len > SWA_NOALLOC_TILE_CAPACITY) break;
    }
    return len;
}

// Thread 0 writes the offsets; then every thread fills the entries of its blocks.
__global__ void noalloc_build_tiles_kernel(int* list, int N, int W, int stride, int rpb) {
    const int nblk = (N + rpb - 1) / rpb;
    if (threadIdx.x == 0) {
        int pos = 0;
        list[0] = 0;
        for (int blk = 0; blk < nblk; ++blk) {
            long long nc, wf, wl;
            noalloc_block_counts(blk, N, W, stride, rpb, &nc, &wf, &wl);
            pos += (int)(nc + (wl - wf + 1));
            list[blk + 1] = pos;
        }
    }
    __syncthreads();
    for (int blk = threadIdx.x; blk < nblk; blk += blockDim.x) {
        long long nc, wf, wl;
        noalloc_block_counts(blk, N, W, stride, rpb, &nc, &wf, &wl);
        int* e = list + nblk + 1 + list[blk];
        for (long long c = 0; c < nc; ++c)
            *e++ = (swa::TILE_KIND_STRIDED << swa::TILE_KIND_SHIFT) | (int)c;
        for (long long t = wf; t <= wl; ++t)
            *e++ = (swa::TILE_KIND_WINDOW << swa::TILE_KIND_SHIFT) | (int)t;
    }
}

// ---------------------------------------------------------------------------------------
// Decode against a rolling cache
// ---------------------------------------------------------------------------------------
size_t decode_part_o_bytes(long long B, long long Hq, long long nsplit, int d) {
    return (size_t)(B * Hq * nsplit * d) * sizeof(float);
}

size_t decode_workspace_bytes(long long B, long long Hq, long long W, int d) {
    const long long nsplit = (W + swa::DEC_KS - 1) / swa::DEC_KS;
    const size_t o = (decode_part_o_bytes(B, Hq, nsplit, d) + 255) / 256 * 256;
    return o + (size_t)(B * Hq * nsplit * 2) * sizeof(float);
}

template <int D, int G>
int launch_decode(const swa::DecParams& dp, int B, int Hkv, cudaStream_t stream, DeviceState& st,
                  int gi) {
    // d = 128: the tensor-core split; d = 64: the CUDA-core split
    constexpr int BYTES = (D == 128) ? swa::DecMmaSmem<G>::BYTES : swa::DecSmem<D, G>::BYTES;
    void (*kern)(const swa::DecParams);
    if constexpr (D == 128)
        kern = swa::decode_mma_kernel<G>;
    else
        kern = swa::decode_split_kernel<D, G>;
    bool& set = st.dec_attr_set[D == 128 ? 1 : 0][gi];
    if (!set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BYTES) !=
            cudaSuccess)
            return SWA_ERR_CUDA;
        set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)dp.nsplit, (unsigned)(B * Hkv), 1);
    cfg.blockDim = dim3(swa::DEC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = BYTES;
    cfg.stream = stream;
    if (cudaLaunchKernelEx(&cfg, kern, dp) != cudaSuccess) return SWA_ERR_CUDA;
    cudaLaunchConfig_t cc = {};
    cc.gridDim = dim3((unsigned)(B * dp.Hq), 1, 1);
    cc.blockDim = dim3((unsigned)D, 1, 1);
    cc.stream = stream;
    return cudaLaunchKernelEx(&cc, swa::decode_combine_kernel<D>, dp) == cudaSuccess ? SWA_OK
                                                                                      : SWA_ERR_CUDA;
}

template <int D>
int dispatch_decode(int g, const swa::DecParams& dp, int B, int Hkv, cudaStream_t stream,
                    DeviceState& st) {
    if (g <= 1) return launch_decode<D, 1>(dp, B, Hkv, stream, st, 0);
    if (g <= 2) return launch_decode<D, 2>(dp, B, Hkv, stream, st, 1);
    if (g <= 4) return launch_decode<D, 4>(dp, B, Hkv, stream, st, 2);
    if (g <= 8) return launch_decode<D, 8>(dp, B, Hkv, stream, st, 3);
    return launch_decode<D, 16>(dp, B, Hkv, stream, st, 4);
}

}  // namespace

namespace {
size_t bwd_workspace_bytes(int B, int Hq, int N) {
    return ((size_t)B * Hq * N * sizeof(float) + 255) / 256 * 256;
}

// The compact keys of the local + strided / global-prefix backward: how many any row reads,
// that count padded to whole tiles, and the query-tile chunks the compact pass is split into
// (about two CTAs per SM of a 148-SM part, at most one chunk per query tile).
struct CompactPlan {
    int ncomp = 0, ncomp_pad = 0, cchunks = 1;
};
CompactPlan compact_plan(int B, int Hkv, int N, int W, int stride, int cap) {
    CompactPlan c;
    if (cap <= 0 || N <= W) return c;
    c.ncomp = (int)std::min<long long>(cap, ((long long)N - W + stride - 1) / stride);
    c.ncomp_pad = (c.ncomp + BN - 1) / BN * BN;
    const long long ctas = (long long)(c.ncomp_pad / BN) * B * Hkv;
    const int n_qtiles = (N + BM - 1) / BM;
    c.cchunks = (int)std::max<long long>(1, std::min<long long>(n_qtiles, (296 + ctas - 1) / ctas));
    return c;
}
size_t compact_part_bytes(const CompactPlan& c, int B, int Hkv, int d) {
    return (size_t)2 * c.cchunks * B * Hkv * c.ncomp_pad * d * sizeof(float);
}

template <int D, int KIND>
int launch_bwd(const swa::BwdParams& bp, int n_tiles, int n_mats, cudaStream_t stream,
               DeviceState& st) {
    using L = swa::BwdLayout<D, KIND == 1 ? 1 : 0>;
    auto kern = swa::attn_bwd_kernel<D, KIND>;
    bool& set = st.bwd_attr_set[D == 128 ? 1 : 0][KIND];
    if (!set) {
        const cudaError_t ea =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
        if (ea != cudaSuccess) return cuda_fail("cudaFuncSetAttribute (backward)", ea);
        set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n_tiles, (unsigned)n_mats, 1);
    cfg.blockDim = dim3(swa::BWD_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::BYTES;
    cfg.stream = stream;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, bp);
    return e == cudaSuccess ? SWA_OK : cuda_fail("cudaLaunchKernelEx (backward)", e);
}

template <int D>
int run_bwd(const swa::BwdParams& bp, const void* out, const void* dout, float* delta,
            cudaStream_t stream, DeviceState& st) {
    const long long rows = (long long)bp.B * bp.Hq * bp.N;
    const int n_tiles = (bp.N + swa::BM - 1) / swa::BM;
    int rc = launch_plain(swa::bwd_delta_kernel<D>, (unsigned)((rows + 255) / 256), 256u, stream,
                          static_cast<const __nv_bfloat16*>(out),
                          static_cast<const __nv_bfloat16*>(dout), delta, rows);
    if (rc) return rc;
    if (bp.cap > 0 && bp.ncomp > 0) {
        if ((rc = launch_bwd<D, 2>(bp, (bp.ncomp_pad / swa::BN) * bp.cchunks, bp.B * bp.Hkv,
                                   stream, st)))
            return rc;
        if (bp.cchunks > 1) {
            const long long slot = (long long)bp.B * bp.Hkv * bp.ncomp_pad * D;
            const unsigned grid = (unsigned)std::min<long long>((2 * slot + 255) / 256, 4096);
            if ((rc = launch_plain(swa::bwd_compact_reduce_kernel, grid, 256u, stream, bp.cpart,
                                   bp.cchunks, slot)))
                return rc;
        }
    }
    if ((rc = launch_bwd<D, 0>(bp, n_tiles, bp.B * bp.Hkv, stream, st))) return rc;
    return launch_bwd<D, 1>(bp, n_tiles, bp.B * bp.Hq, stream, st);
}
}  // namespace

extern "C" {

const char* swa_last_error_detail(void) { return t_err_detail; }

const char* swa_status_string(int status) {
    switch (status) {
        case SWA_OK: return "ok";
        case SWA_ERR_NULL: return "null pointer argument";
        case SWA_ERR_SHAPE: return "invalid shape argument";
        case SWA_ERR_ALIGN: return "pointer not 16-byte aligned";
        case SWA_ERR_UNSUPPORTED: return "unsupported head dimension or device (needs d in {64,128} on sm_103)";
        case SWA_ERR_CUDA: return "CUDA runtime or driver error";
        case SWA_ERR_TIMEOUT: return "kernel watchdog: a bounded wait ran out";
        case SWA_ERR_VALUE: return "invalid scalar argument (scale must be finite and > 0; lambda finite)";
        case SWA_ERR_TOO_LARGE: return "a fixed capacity is too small (the allocation-free tile list, or the decode workspace passed in)";
        default: return "unknown status";
    }
}

int swa_attn_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                     int Hq, int Hkv, int N, int d, int W, float scale, void* stream) {
    if (!q || !k || !v || !out) return SWA_ERR_NULL;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return SWA_ERR_ALIGN;
    if (W < 1) return SWA_ERR_SHAPE;
    int rc = check_common(B, Hq, Hkv, N, d, scale);
    if (rc) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return SWA_ERR_ALIGN;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    if ((rc = current_device_state(&st))) return rc;
    KParams kp;
    std::memset(&kp, 0, sizeof(kp));
    fill_common(kp, B, Hq, Hkv, N, std::min(W, N), 1, scale, out, *st);
    kp.lse = lse;
    kp.pair_mode = ((Hq / Hkv) % 2 == 0) ? 1 : 0;
    if ((rc = make_map(&kp.tm_q, q, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_out, out, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_k, k, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_v, v, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    return dispatch<swa::MODE_WINDOW>(d, kp, n_items_for(kp), static_cast<cudaStream_t>(stream),
                                      *st);
}

int swa_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv,
                 int N, int d, int W, float scale, void* stream) {
    return swa_attn_fwd_lse(q, k, v, out, nullptr, B, Hq, Hkv, N, d, W, scale, stream);
}

int swa_chunk_fwd(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                  int Hkv, int C, int L, int d, int W, float scale, void* stream) {
    if (!q || !k || !v || !out) return SWA_ERR_NULL;
    if (W < 1 || C < 1 || L < C) return SWA_ERR_SHAPE;
    int rc = check_common(B, Hq, Hkv, L, d, scale);
    if (rc) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return SWA_ERR_ALIGN;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    if ((rc = current_device_state(&st))) return rc;
    KParams kp;
    std::memset(&kp, 0, sizeof(kp));
    // queries: C rows; keys: L rows; query row c sits at key position L - C + c
    fill_common(kp, B, Hq, Hkv, C, std::min(W, L), 1, scale, out, *st);
    kp.q_off = L - C;
    kp.pair_mode = ((Hq / Hkv) % 2 == 0) ? 1 : 0;
    if ((rc = make_map(&kp.tm_q, q, d, C, d, (long long)B * Hq, (long long)C * d))) return rc;
    if ((rc = make_map(&kp.tm_out, out, d, C, d, (long long)B * Hq, (long long)C * d))) return rc;
    if ((rc = make_map(&kp.tm_k, k, d, L, d, (long long)B * Hkv, (long long)L * d))) return rc;
    if ((rc = make_map(&kp.tm_v, v, d, L, d, (long long)B * Hkv, (long long)L * d))) return rc;
    return dispatch<swa::MODE_WINDOW>(d, kp, n_items_for(kp), static_cast<cudaStream_t>(stream),
                                      *st);
}

namespace {
// The strided kernel over window tiles plus compact tiles of the keys 0, s, 2s, ... that lie
// before a row's window, at most `cap` of them.
int strided_common(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                   int Hq, int Hkv, int N, int d, int W, int stride, int cap, float scale,
                   void* stream) {
    if (!q || !k || !v || !out) return SWA_ERR_NULL;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return SWA_ERR_ALIGN;
    if (W < 1 || stride < 1) return SWA_ERR_SHAPE;
    int rc = check_common(B, Hq, Hkv, N, d, scale);
    if (rc) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return SWA_ERR_ALIGN;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    if ((rc = current_device_state(&st))) return rc;
    KParams kp;
    std::memset(&kp, 0, sizeof(kp));
    const int Wc = std::min(W, N);
    const int sc = std::min(stride, N);  // a stride >= N opens key 0 only, as stride N does
    fill_common(kp, B, Hq, Hkv, N, Wc, sc, scale, out, *st);
    kp.lse = lse;
    kp.strided_cap = cap;
    kp.pair_mode = ((Hq / Hkv) % 2 == 0) ? 1 : 0;
    const int* list = nullptr;
    if ((rc = get_tile_list(*st, N, Wc, sc, kp.pair_mode ? BM : 2 * BM, cap,
                            static_cast<cudaStream_t>(stream), &list)))
        return rc;
    kp.tiles = list;
    const long long ns = (N - 1) / sc + 1;  // keys 0, s, 2s, ... < N
    if ((rc = make_map(&kp.tm_q, q, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_out, out, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_k, k, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_v, v, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_k2, k, d, ns, (long long)sc * d, (long long)B * Hkv,
                       (long long)N * d)))
        return rc;
    if ((rc = make_map(&kp.tm_v2, v, d, ns, (long long)sc * d, (long long)B * Hkv,
                       (long long)N * d)))
        return rc;
    return dispatch<swa::MODE_STRIDED>(d, kp, n_items_for(kp), static_cast<cudaStream_t>(stream),
                                       *st);
}
}  // namespace

int strided_attn_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse,
                         int B, int Hq, int Hkv, int N, int d, int W, int stride, float scale,
                         void* stream) {
    return strided_common(q, k, v, out, lse, B, Hq, Hkv, N, d, W, stride, 0x7fffffff, scale,
                          stream);
}

int global_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                    int Hkv, int N, int d, int W, int n_global, float scale, void* stream) {
    if (n_global < 0) return SWA_ERR_SHAPE;
    return strided_common(q, k, v, out, nullptr, B, Hq, Hkv, N, d, W, 1, std::min(n_global, N),
                          scale, stream);
}

int strided_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                     int Hkv, int N, int d, int W, int stride, float scale, void* stream) {
    return strided_attn_fwd_lse(q, k, v, out, nullptr, B, Hq, Hkv, N, d, W, stride, scale, stream);
}

int strided_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, int B,
                             int Hq, int Hkv, int N, int d, int W, int stride, float scale,
                             void* stream) {
    if (!q || !k || !v || !out) return SWA_ERR_NULL;
    if (W < 1 || stride < 1) return SWA_ERR_SHAPE;
    int rc = check_common(B, Hq, Hkv, N, d, scale);
    if (rc) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return SWA_ERR_ALIGN;
    const int Wc = std::min(W, N);
    const int sc = std::min(stride, N);
    const int pair_mode = ((Hq / Hkv) % 2 == 0) ? 1 : 0;
    const int rpb = pair_mode ? BM : 2 * BM;
    if (noalloc_list_length(N, Wc, sc, rpb) > SWA_NOALLOC_TILE_CAPACITY) return SWA_ERR_TOO_LARGE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    if ((rc = current_device_state(&st))) return rc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SWA_ERR_CUDA;
    NoAllocState& na = g_noalloc[dev];
    if (!na.ready) {  // once per device, with that device current
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_tiles) != cudaSuccess || ptr == nullptr)
            return SWA_ERR_CUDA;
        na.tiles = static_cast<int*>(ptr);
        na.ready = true;
    }
    // every tensor map is encoded before anything is launched: a call that fails here
    // leaves the shared tile array as the previous call left it
    KParams kp;
    std::memset(&kp, 0, sizeof(kp));
    fill_common(kp, B, Hq, Hkv, N, Wc, sc, scale, out, *st);
    kp.pair_mode = pair_mode;
    kp.tiles = na.tiles;
    const long long ns = (N - 1) / sc + 1;
    if ((rc = make_map(&kp.tm_q, q, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_out, out, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_k, k, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_v, v, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_k2, k, d, ns, (long long)sc * d, (long long)B * Hkv,
                       (long long)N * d)))
        return rc;
    if ((rc = make_map(&kp.tm_v2, v, d, ns, (long long)sc * d, (long long)B * Hkv,
                       (long long)N * d)))
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = s;
        if (cudaLaunchKernelEx(&cfg, noalloc_build_tiles_kernel, na.tiles, N, Wc, sc, rpb) !=
            cudaSuccess)
            return SWA_ERR_CUDA;
    }
    return dispatch<swa::MODE_STRIDED>(d, kp, n_items_for(kp), s, *st);
}

namespace {
int diff_common(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                float lambda, const float* lambda_heads, void* out, int B, int Hq, int Hkv,
                int N, int d, int W, float scale, void* stream) {
    if (!q1 || !k1 || !q2 || !k2 || !v || !out) return SWA_ERR_NULL;
    int rc = check_common(B, Hq, Hkv, N, d, scale);
    if (rc) return rc;
    if (W < 1) return SWA_ERR_SHAPE;
    if (W > N) W = N;
    if (!std::isfinite(lambda)) return SWA_ERR_VALUE;
    if (!aligned16(q1) || !aligned16(k1) || !aligned16(q2) || !aligned16(k2) || !aligned16(v) ||
        !aligned16(out))
        return SWA_ERR_ALIGN;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    if ((rc = current_device_state(&st))) return rc;
    KParams kp;
    std::memset(&kp, 0, sizeof(kp));
    fill_common(kp, B, Hq, Hkv, N, W, 1, scale, out, *st);
    kp.lambda = lambda;
    kp.lambda_heads = lambda_heads;
    kp.pair_mode = 1;  // the two slots are the two score streams of the same rows
    if ((rc = make_map(&kp.tm_q, q1, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_out, out, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_k, k1, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_q2, q2, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_k2, k2, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    if ((rc = make_map(&kp.tm_v, v, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    const int n_items = B * Hq * kp.n_qtiles;
    return dispatch<swa::MODE_DIFF>(d, kp, n_items, static_cast<cudaStream_t>(stream), *st);
}
}  // namespace

int diff_attn_fwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                  float lambda, void* out, int B, int Hq, int Hkv, int N, int d, float scale,
                  void* stream) {
    return diff_common(q1, k1, q2, k2, v, lambda, nullptr, out, B, Hq, Hkv, N, d, N, scale,
                       stream);
}

int diff_attn_fwd_heads(const void* q1, const void* k1, const void* q2, const void* k2,
                        const void* v, const float* lambda, void* out, int B, int Hq, int Hkv,
                        int N, int d, float scale, void* stream) {
    if (!lambda) return SWA_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(lambda) & 3u) != 0) return SWA_ERR_ALIGN;
    return diff_common(q1, k1, q2, k2, v, 0.f, lambda, out, B, Hq, Hkv, N, d, N, scale, stream);
}

int diff_swa_attn_fwd(const void* q1, const void* k1, const void* q2, const void* k2,
                      const void* v, float lambda, const float* lambda_heads, void* out, int B,
                      int Hq, int Hkv, int N, int d, int W, float scale, void* stream) {
    if (lambda_heads && (reinterpret_cast<uintptr_t>(lambda_heads) & 3u) != 0)
        return SWA_ERR_ALIGN;
    return diff_common(q1, k1, q2, k2, v, lambda_heads ? 0.f : lambda, lambda_heads, out, B, Hq,
                       Hkv, N, d, W, scale, stream);
}

int swa_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SWA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = current_device_state(&st);
    if (rc) return rc;
    int word = 0;
    if (cudaMemcpy(&word, st->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SWA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(st->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
        return SWA_ERR_CUDA;
    return word == 0 ? SWA_OK : word;
}

int swa_watchdog_selftest(int limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 1000000) return SWA_ERR_VALUE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = current_device_state(&st);
    if (rc) return rc;
    return launch_plain(swa::watchdog_selftest_kernel, 1u, 32u, static_cast<cudaStream_t>(stream),
                        st->status, (unsigned long long)limit_us * 1000ull);
}

size_t swa_decode_workspace_bytes(int B, int Hq, int W, int d) {
    if (B < 1 || Hq < 1 || W < 1 || (d != 64 && d != 128)) return 0;
    return decode_workspace_bytes(B, Hq, W, d);
}

int swa_decode_fwd(const void* q, const void* k_cache, const void* v_cache, const int* pos,
                   void* out, int B, int Hq, int Hkv, int W, int d, float scale, void* workspace,
                   size_t workspace_bytes, void* stream) {
    if (!q || !k_cache || !v_cache || !pos || !out || !workspace) return SWA_ERR_NULL;
    if (B < 1 || Hq < 1 || Hkv < 1 || W < 1 || Hq % Hkv != 0) return SWA_ERR_SHAPE;
    if ((long long)B * Hkv > 65535 || (long long)B * Hq > (1ll << 24) || W > (1 << 30))
        return SWA_ERR_SHAPE;
    if (d != 64 && d != 128) return SWA_ERR_UNSUPPORTED;
    if (Hq / Hkv > 16) return SWA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale) || !(scale > 0.f)) return SWA_ERR_VALUE;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
        (reinterpret_cast<uintptr_t>(pos) & 3u) != 0)
        return SWA_ERR_ALIGN;
    if (workspace_bytes < decode_workspace_bytes(B, Hq, W, d)) return SWA_ERR_TOO_LARGE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = current_device_state(&st);
    if (rc) return rc;
    swa::DecParams dp;
    std::memset(&dp, 0, sizeof(dp));
    const long long nsplit = (W + swa::DEC_KS - 1) / swa::DEC_KS;
    if ((rc = make_map(&dp.tm_kc, k_cache, d, W, d, (long long)B * Hkv, (long long)W * d,
                       swa::DEC_KS)))
        return rc;
    if ((rc = make_map(&dp.tm_vc, v_cache, d, W, d, (long long)B * Hkv, (long long)W * d,
                       swa::DEC_KS)))
        return rc;
    dp.q = static_cast<const __nv_bfloat16*>(q);
    dp.pos = pos;
    dp.out = static_cast<__nv_bfloat16*>(out);
    dp.part_o = static_cast<float*>(workspace);
    dp.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          (decode_part_o_bytes(B, Hq, nsplit, d) + 255) / 256 * 256);
    dp.status = st->status;
    dp.wait_limit_ns = kWaitLimitNs;
    dp.B = B;
    dp.Hq = Hq;
    dp.Hkv = Hkv;
    dp.W = W;
    dp.nsplit = (int)nsplit;
    dp.scale_log2 = scale * 1.4426950408889634f;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d == 128) return dispatch_decode<128>(Hq / Hkv, dp, B, Hkv, s, *st);
    return dispatch_decode<64>(Hq / Hkv, dp, B, Hkv, s, *st);
}


size_t swa_attn_bwd_workspace_bytes(int B, int Hq, int N) {
    if (B < 1 || Hq < 1 || N < 1) return 0;
    return bwd_workspace_bytes(B, Hq, N);
}

namespace {
// The backward of the window mask and of its local + strided / global-prefix extensions:
// cap = 0 is the plain window; otherwise row i also reads the keys r * stride with
// r < min(ceil(lo(i) / stride), cap).
int bwd_common(const void* q, const void* k, const void* v, const void* out, const float* lse,
               const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
               int d, int W, int stride, int cap, float scale, void* workspace,
               size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv || !workspace)
        return SWA_ERR_NULL;
    int rc = check_common(B, Hq, Hkv, N, d, scale);
    if (rc) return rc;
    if (W < 1 || stride < 1 || cap < 0) return SWA_ERR_SHAPE;
    if (W > N) W = N;
    if (stride > N) stride = N;  // a stride >= N reaches key 0 only, as stride N does
    // grid: (row tiles, heads); the second grid dimension is at most 65535
    if ((long long)B * Hq > 65535 || (long long)B * Hq * N > (1ll << 38)) return SWA_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
        return SWA_ERR_ALIGN;
    const CompactPlan cp = compact_plan(B, Hkv, N, W, stride, cap);
    const size_t delta_bytes = bwd_workspace_bytes(B, Hq, N);
    if (workspace_bytes < delta_bytes + compact_part_bytes(cp, B, Hkv, d)) return SWA_ERR_TOO_LARGE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    if ((rc = current_device_state(&st))) return rc;
    swa::BwdParams bp;
    std::memset(&bp, 0, sizeof(bp));
    if ((rc = make_map(&bp.tm_q, q, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&bp.tm_do, dout, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&bp.tm_k, k, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    if ((rc = make_map(&bp.tm_v, v, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    if (cap > 0) {
        const long long ns = (N - 1) / stride + 1;  // keys 0, s, 2s, ... < N
        if ((rc = make_map(&bp.tm_k2, k, d, ns, (long long)stride * d, (long long)B * Hkv,
                           (long long)N * d)))
            return rc;
        if ((rc = make_map(&bp.tm_v2, v, d, ns, (long long)stride * d, (long long)B * Hkv,
                           (long long)N * d)))
            return rc;
    }
    bp.lse = lse;
    bp.delta = static_cast<const float*>(workspace);
    bp.dq = static_cast<__nv_bfloat16*>(dq);
    bp.dk = static_cast<__nv_bfloat16*>(dk);
    bp.dv = static_cast<__nv_bfloat16*>(dv);
    bp.cpart = reinterpret_cast<float*>(static_cast<char*>(workspace) + delta_bytes);
    bp.status = st->status;
    bp.wait_limit_ns = kWaitLimitNs;
    bp.B = B;
    bp.Hq = Hq;
    bp.Hkv = Hkv;
    bp.N = N;
    bp.W = W;
    bp.stride = stride;
    bp.cap = cap;
    bp.ncomp = cp.ncomp;
    bp.ncomp_pad = cp.ncomp_pad;
    bp.cchunks = cp.cchunks;
    bp.scale = scale;
    bp.scale_log2 = scale * 1.4426950408889634f;
    float* delta = static_cast<float*>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d == 128) return run_bwd<128>(bp, out, dout, delta, s, *st);
    return run_bwd<64>(bp, out, dout, delta, s, *st);
}
}  // namespace

size_t diff_attn_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || (d != 64 && d != 128)) return 0;
    return 2 * bwd_workspace_bytes(B, Hq, N) + (size_t)B * Hkv * N * d * sizeof(float);
}

int diff_attn_bwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                  float lambda, const float* lambda_heads, const void* out1, const float* lse1,
                  const void* out2, const float* lse2, const void* dout, void* dq1, void* dk1,
                  void* dq2, void* dk2, void* dv, float* dlambda, int B, int Hq, int Hkv, int N,
                  int d, int W, float scale, void* workspace, size_t workspace_bytes,
                  void* stream) {
    if (!q1 || !k1 || !q2 || !k2 || !v || !out1 || !lse1 || !out2 || !lse2 || !dout || !dq1 ||
        !dk1 || !dq2 || !dk2 || !dv || !workspace)
        return SWA_ERR_NULL;
    int rc = check_common(B, Hq, Hkv, N, d, scale);
    if (rc) return rc;
    if (W < 1) return SWA_ERR_SHAPE;
    if (W > N) W = N;
    if (!lambda_heads && !std::isfinite(lambda)) return SWA_ERR_VALUE;
    if ((long long)B * Hq > 65535 || (long long)B * Hq * N > (1ll << 38)) return SWA_ERR_SHAPE;
    const void* al16[] = {q1, k1, q2, k2, v, out1, out2, dout, dq1, dk1, dq2, dk2, dv, workspace};
    for (const void* ptr : al16)
        if (!aligned16(ptr)) return SWA_ERR_ALIGN;
    for (const void* ptr : {static_cast<const void*>(lse1), static_cast<const void*>(lse2),
                            static_cast<const void*>(lambda_heads), static_cast<const void*>(dlambda)})
        if (ptr && (reinterpret_cast<uintptr_t>(ptr) & 3u) != 0) return SWA_ERR_ALIGN;
    if (workspace_bytes < diff_attn_bwd_workspace_bytes(B, Hq, Hkv, N, d)) return SWA_ERR_TOO_LARGE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    if ((rc = current_device_state(&st))) return rc;
    // workspace: delta of map 1, delta of map 2, dV of map 1 (fp32)
    const size_t db = bwd_workspace_bytes(B, Hq, N);
    float* delta1 = static_cast<float*>(workspace);
    float* delta2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + db);
    float* dv32 = reinterpret_cast<float*>(static_cast<char*>(workspace) + 2 * db);
    swa::BwdParams p1;
    std::memset(&p1, 0, sizeof(p1));
    swa::BwdParams p2;
    std::memset(&p2, 0, sizeof(p2));
    if ((rc = make_map(&p1.tm_q, q1, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&p1.tm_k, k1, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    if ((rc = make_map(&p1.tm_v, v, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    if ((rc = make_map(&p1.tm_do, dout, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&p2.tm_q, q2, d, N, d, (long long)B * Hq, (long long)N * d))) return rc;
    if ((rc = make_map(&p2.tm_k, k2, d, N, d, (long long)B * Hkv, (long long)N * d))) return rc;
    p2.tm_v = p1.tm_v;
    p2.tm_do = p1.tm_do;
    for (swa::BwdParams* bp : {&p1, &p2}) {
        bp->status = st->status;
        bp->wait_limit_ns = kWaitLimitNs;
        bp->B = B;
        bp->Hq = Hq;
        bp->Hkv = Hkv;
        bp->N = N;
        bp->W = W;
        bp->stride = 1;
        bp->cap = 0;
        bp->cchunks = 1;
        bp->scale = scale;
        bp->scale_log2 = scale * 1.4426950408889634f;
        bp->dv = static_cast<__nv_bfloat16*>(dv);
    }
    p1.lse = lse1;
    p1.delta = delta1;
    p1.dq = static_cast<__nv_bfloat16*>(dq1);
    p1.dk = static_cast<__nv_bfloat16*>(dk1);
    p1.dv32_out = dv32;
    p2.lse = lse2;
    p2.delta = delta2;
    p2.dq = static_cast<__nv_bfloat16*>(dq2);
    p2.dk = static_cast<__nv_bfloat16*>(dk2);
    p2.dv32_in = dv32;
    p2.mu_mode = 1;
    p2.lam = lambda_heads ? 0.f : lambda;
    p2.lam_heads = lambda_heads;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long rows = (long long)B * Hq * N;
    const unsigned dgrid = (unsigned)((rows + 255) / 256);
    const int n_tiles = (N + BM - 1) / BM;
    auto run = [&](auto dtag) -> int {
        constexpr int D = decltype(dtag)::value;
        const auto* go = static_cast<const __nv_bfloat16*>(dout);
        int r;
        if ((r = launch_plain(swa::bwd_delta_kernel<D>, dgrid, 256u, s,
                              static_cast<const __nv_bfloat16*>(out1), go, delta1, rows)))
            return r;
        if ((r = launch_plain(swa::bwd_delta_kernel<D>, dgrid, 256u, s,
                              static_cast<const __nv_bfloat16*>(out2), go, delta2, rows)))
            return r;
        if ((r = launch_bwd<D, 0>(p1, n_tiles, B * Hkv, s, *st))) return r;  // dk1, dV1 (fp32)
        if ((r = launch_bwd<D, 0>(p2, n_tiles, B * Hkv, s, *st))) return r;  // dk2, dv
        if ((r = launch_bwd<D, 1>(p1, n_tiles, B * Hq, s, *st))) return r;   // dq1
        if ((r = launch_bwd<D, 1>(p2, n_tiles, B * Hq, s, *st))) return r;   // dq2
        if (dlambda &&
            (r = launch_plain(swa::bwd_dlam_kernel, (unsigned)Hq, 256u, s,
                              static_cast<const float*>(delta2), dlambda, B, Hq, N)))
            return r;
        return SWA_OK;
    };
    if (d == 128) return run(std::integral_constant<int, 128>{});
    return run(std::integral_constant<int, 64>{});
}

int swa_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                 int d, int W, float scale, void* workspace, size_t workspace_bytes,
                 void* stream) {
    return bwd_common(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, W, 1, 0, scale,
                      workspace, workspace_bytes, stream);
}

size_t strided_attn_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int W,
                                        int stride) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || W < 1 || stride < 1 || (d != 64 && d != 128))
        return 0;
    const CompactPlan cp = compact_plan(B, Hkv, N, std::min(W, N), std::min(stride, N), 0x7fffffff);
    return bwd_workspace_bytes(B, Hq, N) + compact_part_bytes(cp, B, Hkv, d);
}

int strided_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                     int Hq, int Hkv, int N, int d, int W, int stride, float scale,
                     void* workspace, size_t workspace_bytes, void* stream) {
    if (stride < 1) return SWA_ERR_SHAPE;
    return bwd_common(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, W, stride,
                      0x7fffffff, scale, workspace, workspace_bytes, stream);
}

size_t global_attn_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int W,
                                       int n_global) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || W < 1 || n_global < 0 || (d != 64 && d != 128))
        return 0;
    const CompactPlan cp = compact_plan(B, Hkv, N, std::min(W, N), 1, std::min(n_global, N));
    return bwd_workspace_bytes(B, Hq, N) + compact_part_bytes(cp, B, Hkv, d);
}

int global_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                    const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                    int Hq, int Hkv, int N, int d, int W, int n_global, float scale,
                    void* workspace, size_t workspace_bytes, void* stream) {
    if (n_global < 0) return SWA_ERR_SHAPE;
    return bwd_common(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, W, 1,
                      std::min(n_global, std::max(N, 1)), scale, workspace, workspace_bytes,
                      stream);
}

int global_attn_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse,
                        int B, int Hq, int Hkv, int N, int d, int W, int n_global, float scale,
                        void* stream) {
    if (n_global < 0) return SWA_ERR_SHAPE;
    return strided_common(q, k, v, out, lse, B, Hq, Hkv, N, d, W, 1,
                          std::min(n_global, std::max(N, 1)), scale, stream);
}

int swa_cache_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                     const int* pos, int B, int Hkv, int W, int d, int n, void* stream) {
    if (!k_new || !v_new || !k_cache || !v_cache || !pos) return SWA_ERR_NULL;
    if (B < 1 || Hkv < 1 || W < 1 || n < 1 || (long long)B * Hkv > (1ll << 30)) return SWA_ERR_SHAPE;
    if (d != 64 && d != 128) return SWA_ERR_UNSUPPORTED;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(pos) & 3u) != 0)
        return SWA_ERR_ALIGN;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = current_device_state(&st);
    if (rc) return rc;
    // rows on gridDim.x (up to 2^31 - 1), (sequence, KV head) pairs on gridDim.y (at most
    // 65535 blocks, the kernel strides over the rest)
    const int n_bh = B * Hkv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min(n, W), (unsigned)std::min(n_bh, 65535), 1);
    cfg.blockDim = dim3((unsigned)(d / 8), 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    const auto* kn = static_cast<const __nv_bfloat16*>(k_new);
    const auto* vn = static_cast<const __nv_bfloat16*>(v_new);
    auto* kc = static_cast<__nv_bfloat16*>(k_cache);
    auto* vc = static_cast<__nv_bfloat16*>(v_cache);
    cudaError_t e = (d == 128)
        ? cudaLaunchKernelEx(&cfg, swa::cache_append_kernel<128>, kn, vn, kc, vc, pos, n_bh, Hkv, W, n)
        : cudaLaunchKernelEx(&cfg, swa::cache_append_kernel<64>, kn, vn, kc, vc, pos, n_bh, Hkv, W, n);
    return e == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

int swa_cache_gather(const void* k_cache, const void* v_cache, void* k_ctx, void* v_ctx, int B,
                     int Hkv, int W, int d, int pos0, int nctx, int ctx_rows, void* stream) {
    if (!k_cache || !v_cache || !k_ctx || !v_ctx) return SWA_ERR_NULL;
    if (B < 1 || Hkv < 1 || W < 1 || nctx < 0 || nctx > W || nctx > pos0 || ctx_rows < nctx ||
        (long long)B * Hkv > (1ll << 30))
        return SWA_ERR_SHAPE;
    if (d != 64 && d != 128) return SWA_ERR_UNSUPPORTED;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_ctx) || !aligned16(v_ctx))
        return SWA_ERR_ALIGN;
    if (nctx == 0) return SWA_OK;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    int rc = current_device_state(&st);
    if (rc) return rc;
    const int n_bh = B * Hkv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nctx, (unsigned)std::min(n_bh, 65535), 1);
    cfg.blockDim = dim3((unsigned)(d / 8), 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    const auto* kc = static_cast<const __nv_bfloat16*>(k_cache);
    const auto* vc = static_cast<const __nv_bfloat16*>(v_cache);
    auto* kx = static_cast<__nv_bfloat16*>(k_ctx);
    auto* vx = static_cast<__nv_bfloat16*>(v_ctx);
    cudaError_t e = (d == 128)
        ? cudaLaunchKernelEx(&cfg, swa::cache_gather_kernel<128>, kc, vc, kx, vx, n_bh, W, pos0, nctx, ctx_rows)
        : cudaLaunchKernelEx(&cfg, swa::cache_gather_kernel<64>, kc, vc, kx, vx, n_bh, W, pos0, nctx, ctx_rows);
    return e == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

}  // extern "C"
