// decode.cuh -- sm_103a decode step of causal sliding-window attention against a rolling
// W-slot KV cache: one new query per sequence and head.
//
// What it computes ("SWA：滑动窗口注意力与跨层信息传递" §3.1 and §4.2): the key and value
// of absolute position j sit in cache slot j mod W, so the window max(0, t-W+1) .. t of a
// query at position t is exactly the set of slots 0 .. min(t, W-1).  The softmax over a
// set does not depend on the order of its members (positions are already encoded in the
// cached keys), so the kernel reads those slots in slot order.
//
// The step is bound by HBM: every window key and value row is read once and each feeds
// Hq/Hkv queries only.  Split-K over the slots:
//   decode_mma_kernel<G>        d = 128: the same split with both products on tcgen05 (the
//                               slots as the 128 MMA rows, the heads as N = 16 columns); see
//                               below.
//   decode_split_kernel<D, G>   d = 64: grid (splits of DEC_KS slots, B*Hkv), DEC_KS threads.  TMA
//                               loads the split's K and V rows (128B-swizzled boxes) into
//                               shared memory; thread t scores slot t against the G query
//                               heads of the KV head (packed fp32x2 products on the CUDA
//                               cores), the CTA forms max / exp2 / sum per head, then warp w
//                               accumulates the output columns over slots 32w .. 32w+31
//                               (lane l: CPL adjacent columns) and the warps' sums are added.
//                               Writes the split's un-normalised O, its maximum (log2
//                               domain) and its sum l.
//   decode_combine_kernel<D>    grid (B*Hq), D threads: rescales the splits to a common
//                               maximum, out = sum O_s 2^(m_s - m) / sum l_s 2^(m_s - m).
// The CUDA-core products of decode_split_kernel keep a split busy long after its load has
// landed, and only three splits fit on an SM, so too few bytes are in flight; on the tensor
// core the products take a few hundred cycles although 15 of the 16 columns are padding at
// G = 1.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace swa {

constexpr int DEC_KS = 128;  // cache slots per split, one thread per slot (and MMA row)
constexpr int DEC_THREADS = DEC_KS;
constexpr int DEC_WARPS = DEC_KS / 32;

struct DecParams {
    CUtensorMap tm_kc;   // k cache, view [B*Hkv][W][d]
    CUtensorMap tm_vc;   // v cache, view [B*Hkv][W][d]
    const __nv_bfloat16* q;  // [B, Hq, d]
    const int* pos;          // [B] absolute position of each sequence's query (device)
    __nv_bfloat16* out;      // [B, Hq, d]
    float* part_o;           // [B*Hq][nsplit][d] un-normalised split outputs
    float* part_ml;          // [B*Hq][nsplit][2]: split maximum (log2 domain), split sum
    int* status;
    unsigned long long wait_limit_ns;
    int B, Hq, Hkv, W, nsplit;
    float scale_log2;        // scale * log2(e)
};

template <int D, int G>
struct DecSmem {
    static constexpr int KV_BYTES = DEC_KS * D * 2;   // one K or V split, D/64 boxes
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = KV_BYTES;
    static constexpr int OFF_Q = 2 * KV_BYTES;                 // fp32 [G][D]
    static constexpr int OFF_P = OFF_Q + G * D * 4;            // fp32 [G][DEC_KS]
    static constexpr int OFF_RED = OFF_P + G * DEC_KS * 4;     // fp32 [2][DEC_WARPS][G]
    static constexpr int OFF_BAR = OFF_RED + 2 * DEC_WARPS * G * 4;  // two mbarriers (K, V)
    static constexpr int OFF_ABORT = OFF_BAR + 16;
    static constexpr int END = OFF_ABORT + 4;
    static constexpr int BYTES = END + 1024;  // slack for aligning the base to 1024
    static_assert(KV_BYTES % 1024 == 0, "1024-byte box alignment");
    static_assert(DEC_WARPS * G * D * 4 <= 2 * KV_BYTES, "the cross-warp sums fit in the tiles");
};

// Shared-memory byte offset of element (row r, column c) of a DEC_KS-row tile stored as D/64
// boxes of 64 columns, 128 bytes per row, 16-byte unit u of a row at u ^ (r & 7).
__device__ __forceinline__ uint32_t swz_offset(int r, int c) {
    const int box = c >> 6, u = (c & 63) >> 3, e = c & 7;
    return (uint32_t)(box * (DEC_KS * 128) + r * 128 + ((u ^ (r & 7)) << 4) + e * 2);
}

__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
    // the bf16 bits are the high half of the fp32 bits
    return f32x2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <int D, int G>
__global__ void __launch_bounds__(DEC_THREADS) decode_split_kernel(const __grid_constant__ DecParams p) {
    using L = DecSmem<D, G>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    float* qs = reinterpret_cast<float*>(smem + L::OFF_Q);
    float* ps = reinterpret_cast<float*>(smem + L::OFF_P);
    float* red = reinterpret_cast<float*>(smem + L::OFF_RED);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_ABORT);
    const uint32_t bar_k = sbase + L::OFF_BAR, bar_v = bar_k + 8;

    const int split = blockIdx.x;
    const int bh = blockIdx.y;  // b * Hkv + hk
    const int b = bh / p.Hkv, hk = bh % p.Hkv;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int posb = p.pos[b];
    const int nvalid = posb < 0 ? 0 : min(posb + 1, p.W);
    const int k0 = split * DEC_KS;
    if (k0 >= nvalid) return;  // the combine reads only the splits that hold window keys
    const int nk = min(DEC_KS, nvalid - k0);

    if (t == 0) {
        mbar_init(bar_k, 1);
        mbar_init(bar_v, 1);
        *abort_flag = 0;
        fence_barrier_init();
        mbar_arrive_expect_tx(bar_k, L::KV_BYTES);
        for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sbase + L::OFF_K + c * (DEC_KS * 128), &p.tm_kc, bar_k, c * 64, k0, bh);
        mbar_arrive_expect_tx(bar_v, L::KV_BYTES);
        for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sbase + L::OFF_V + c * (DEC_KS * 128), &p.tm_vc, bar_v, c * 64, k0, bh);
    }
    // the g <= G query heads of this KV head, widened to fp32 (rows h >= g are zero)
    const int g = p.Hq / p.Hkv;
    for (int i = t; i < G * (D / 8); i += DEC_THREADS) {
        const int h = i / (D / 8), u = i % (D / 8);
        uint4 raw = make_uint4(0u, 0u, 0u, 0u);
        if (h < g)
            raw = *reinterpret_cast<const uint4*>(p.q + ((size_t)b * p.Hq + (size_t)hk * g + h) * D +
                                                  u * 8);
        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
        float4* dst = reinterpret_cast<float4*>(qs + h * D + u * 8);
        dst[0] = make_float4(__uint_as_float(w4[0] << 16), __uint_as_float(w4[0] & 0xffff0000u),
                             __uint_as_float(w4[1] << 16), __uint_as_float(w4[1] & 0xffff0000u));
        dst[1] = make_float4(__uint_as_float(w4[2] << 16), __uint_as_float(w4[2] & 0xffff0000u),
                             __uint_as_float(w4[3] << 16), __uint_as_float(w4[3] & 0xffff0000u));
    }
    __syncthreads();

    // ---- scores of slot k0 + t against the G heads (log2 domain); two packed partial sums
    // per head keep the dependent chains short
    bool ok = mbar_wait_bounded(bar_k, 0, abort_flag, p.wait_limit_ns);
    float s[G];
    {
        uint64_t sa[G], sb[G];
#pragma unroll
        for (int h = 0; h < G; ++h) sa[h] = sb[h] = 0ull;
        if (ok) {
#pragma unroll 4
            for (int u = 0; u < D / 8; ++u) {
                const uint4 kv = *reinterpret_cast<const uint4*>(smem + L::OFF_K + swz_offset(t, u * 8));
                const uint64_t k0p = bf16x2_to_f32x2(kv.x), k1p = bf16x2_to_f32x2(kv.y);
                const uint64_t k2p = bf16x2_to_f32x2(kv.z), k3p = bf16x2_to_f32x2(kv.w);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const uint4 qa = *reinterpret_cast<const uint4*>(qs + h * D + u * 8);
                    const uint4 qb = *reinterpret_cast<const uint4*>(qs + h * D + u * 8 + 4);
                    sa[h] = f32x2_fma(k0p, (uint64_t)qa.x | ((uint64_t)qa.y << 32), sa[h]);
                    sb[h] = f32x2_fma(k1p, (uint64_t)qa.z | ((uint64_t)qa.w << 32), sb[h]);
                    sa[h] = f32x2_fma(k2p, (uint64_t)qb.x | ((uint64_t)qb.y << 32), sa[h]);
                    sb[h] = f32x2_fma(k3p, (uint64_t)qb.z | ((uint64_t)qb.w << 32), sb[h]);
                }
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float a0, a1, b0, b1;
            f32x2_unpack(sa[h], a0, a1);
            f32x2_unpack(sb[h], b0, b1);
            s[h] = (a0 + a1) + (b0 + b1);
        }
    }
    const bool valid = t < nk;
#pragma unroll
    for (int h = 0; h < G; ++h) s[h] = valid ? s[h] * p.scale_log2 : -INFINITY;

    // ---- per head: maximum and sum over the split (warp shuffles, then the warps)
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float v = s[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) red[warp * G + h] = v;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float mh = red[h];
#pragma unroll
        for (int w = 1; w < DEC_WARPS; ++w) mh = fmaxf(mh, red[w * G + h]);
        const float e = valid ? exp2f(s[h] - mh) : 0.f;
        ps[h * DEC_KS + t] = e;
        float v = e;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[DEC_WARPS * G + warp * G + h] = v;
    }
    if (ok) ok = mbar_wait_bounded(bar_v, 0, abort_flag, p.wait_limit_ns);
    __syncthreads();

    // ---- output columns: warp w takes the split's slots 32w .. 32w+31 and lane l the
    // columns CPL*l .. CPL*l+CPL-1 (one 8- or 4-byte shared load of a V row per slot); the
    // warps' partial sums then meet in shared memory (over the K and V tiles)
    constexpr int CPL = D / 32;  // columns per lane: 4 (D = 128) or 2 (D = 64)
    uint64_t acc[G][CPL / 2];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int j = 0; j < CPL / 2; ++j) acc[h][j] = 0ull;
    if (ok) {
        // only the slots that hold window keys: the others may hold anything, even NaN
        const int kb = warp * 32, ke = min(kb + 32, nk);
        const int c0 = lane * CPL;
        int k = kb;
        for (; k + 4 <= ke; k += 4) {
            uint64_t v2[4][CPL / 2];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint8_t* src = smem + L::OFF_V + swz_offset(k + j, c0);
                if (CPL == 4) {
                    const uint2 u2 = *reinterpret_cast<const uint2*>(src);
                    v2[j][0] = bf16x2_to_f32x2(u2.x);
                    v2[j][CPL / 2 - 1] = bf16x2_to_f32x2(u2.y);
                } else {
                    v2[j][0] = bf16x2_to_f32x2(*reinterpret_cast<const uint32_t*>(src));
                }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float4 pw = *reinterpret_cast<const float4*>(ps + h * DEC_KS + k);
                const float pj[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint64_t pp = f32x2_pack(pj[j], pj[j]);
#pragma unroll
                    for (int c = 0; c < CPL / 2; ++c) acc[h][c] = f32x2_fma(pp, v2[j][c], acc[h][c]);
                }
            }
        }
        for (; k < ke; ++k) {
            const uint8_t* src = smem + L::OFF_V + swz_offset(k, c0);
            uint64_t v2[CPL / 2];
            if (CPL == 4) {
                const uint2 u2 = *reinterpret_cast<const uint2*>(src);
                v2[0] = bf16x2_to_f32x2(u2.x);
                v2[CPL / 2 - 1] = bf16x2_to_f32x2(u2.y);
            } else {
                v2[0] = bf16x2_to_f32x2(*reinterpret_cast<const uint32_t*>(src));
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const uint64_t pp = f32x2_pack(ps[h * DEC_KS + k], ps[h * DEC_KS + k]);
#pragma unroll
                for (int c = 0; c < CPL / 2; ++c) acc[h][c] = f32x2_fma(pp, v2[c], acc[h][c]);
            }
        }
    }
    // warps -> one: partial sums through shared memory (over the K and V tiles)
    float* xs = reinterpret_cast<float*>(smem + L::OFF_K);  // [DEC_WARPS][G][D]
    __syncthreads();  // every thread is done reading the K and V tiles
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int c = 0; c < CPL / 2; ++c) {
            float lo, hi;
            f32x2_unpack(acc[h][c], lo, hi);
            xs[(warp * G + h) * D + lane * CPL + 2 * c] = lo;
            xs[(warp * G + h) * D + lane * CPL + 2 * c + 1] = hi;
        }
    __syncthreads();
    for (int i = t; i < G * D; i += DEC_THREADS) {
        const int h = i / D, c = i % D;
        if (h >= g) break;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < DEC_WARPS; ++w) o += xs[(w * G + h) * D + c];
        const size_t row = ((size_t)b * p.Hq + (size_t)hk * g + h) * p.nsplit + split;
        p.part_o[row * D + c] = o;
        if (c == 0) {
            float l = 0.f, mh = -INFINITY;
#pragma unroll
            for (int w = 0; w < DEC_WARPS; ++w) {
                l += red[DEC_WARPS * G + w * G + h];
                mh = fmaxf(mh, red[w * G + h]);
            }
            p.part_ml[row * 2] = mh;
            p.part_ml[row * 2 + 1] = l;
        }
    }
    if (t == 0 && *abort_flag) atomicExch(p.status, 6 /* SWA_ERR_TIMEOUT */);
}

// ------------------------------------------------------------------------------------------
// Tensor-core form of a split (d = 128).  The slots are the 128 rows of two tcgen05 products
// and the G <= 16 query heads of the KV head their N = 16 columns:
//   S^T[slot][h] = K Q^T   (A: the K tile, K-major; B: the heads' queries, K-major)
//   O^T[c][h]    = V^T P^T (A: the V tile read MN-major; B: the weights, K-major)
// both accumulated in tensor memory (columns [0,16) and [16,32) of a 32-column allocation).
// Thread t owns slot t (TMEM lane t) for the softmax, as in decode_split_kernel, and column
// t of the output afterwards.  Only the softmax stays on the CUDA cores, so a split's life
// is mostly its TMA load.  The weights are rounded to bf16 for the second product (the
// forward kernel does the same); the sum l adds them unrounded.
template <int G>
struct DecMmaSmem {
    static constexpr int D = 128;
    static constexpr int NB = 16;                     // MMA N: the heads, padded
    static constexpr int KV_BYTES = DEC_KS * D * 2;   // a K or V split: two 64-column boxes
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = KV_BYTES;
    static constexpr int OFF_Q = 2 * KV_BYTES;        // bf16 [NB][D], K-major, 128B-swizzled
    static constexpr int OFF_P = OFF_Q + NB * D * 2;  // bf16 [NB][DEC_KS], same layout
    static constexpr int OFF_RED = OFF_P + NB * DEC_KS * 2;          // fp32 [2][DEC_WARPS][G]
    static constexpr int OFF_BAR = OFF_RED + 2 * DEC_WARPS * G * 4;  // K, V, MMA done
    static constexpr int OFF_TMEM = OFF_BAR + 24;
    static constexpr int OFF_ABORT = OFF_TMEM + 4;
    static constexpr int END = OFF_ABORT + 4;
    static constexpr int BYTES = END + 1024;  // slack for aligning the base to 1024
    static constexpr uint32_t TMEM_COLS = 32;
    static_assert(DEC_KS == 128 && DEC_THREADS == 128, "one slot per thread and TMEM lane");
    static_assert(G <= NB, "at most 16 query heads per KV head");
};

// Byte offset of element (row n, column k) of a K-major, 128-byte-swizzled operand tile of
// `rows` rows (a multiple of 8): 64-column chunks of rows x 128 bytes, the 16-byte unit u of
// a row stored at u ^ (n & 7).
__device__ __forceinline__ uint32_t kmajor_sw128(int rows, int n, int k) {
    return (uint32_t)((k >> 6) * (rows * 128) + n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) +
                      (k & 7) * 2);
}

template <int G>
__global__ void __launch_bounds__(DEC_THREADS) decode_mma_kernel(const __grid_constant__ DecParams p) {
    constexpr int D = 128;
    using L = DecMmaSmem<G>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    float* red = reinterpret_cast<float*>(smem + L::OFF_RED);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_ABORT);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM);
    const uint32_t bar_k = sbase + L::OFF_BAR, bar_v = bar_k + 8, bar_m = bar_k + 16;

    const int split = blockIdx.x;
    const int bh = blockIdx.y;  // b * Hkv + hk
    const int b = bh / p.Hkv, hk = bh % p.Hkv;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const uint64_t lim = p.wait_limit_ns;
    const int posb = p.pos[b];
    const int nvalid = posb < 0 ? 0 : min(posb + 1, p.W);
    const int k0 = split * DEC_KS;
    if (k0 >= nvalid) return;  // the combine reads only the splits that hold window keys
    const int nk = min(DEC_KS, nvalid - k0);

    if (t == 0) {
        mbar_init(bar_k, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_m, 1);
        *abort_flag = 0;
        fence_barrier_init();
        mbar_arrive_expect_tx(bar_k, L::KV_BYTES);
        for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sbase + L::OFF_K + c * (DEC_KS * 128), &p.tm_kc, bar_k, c * 64, k0, bh);
        mbar_arrive_expect_tx(bar_v, L::KV_BYTES);
        for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sbase + L::OFF_V + c * (DEC_KS * 128), &p.tm_vc, bar_v, c * 64, k0, bh);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish();
    }
    // the g <= G query heads of this KV head as rows of the B operand (rows h >= g zero)
    const int g = p.Hq / p.Hkv;
    for (int i = t; i < L::NB * (D / 8); i += DEC_THREADS) {
        const int h = i / (D / 8), u = i % (D / 8);
        uint4 raw = make_uint4(0u, 0u, 0u, 0u);
        if (h < g)
            raw = *reinterpret_cast<const uint4*>(p.q + ((size_t)b * p.Hq + (size_t)hk * g + h) * D +
                                                  u * 8);
        *reinterpret_cast<uint4*>(smem + L::OFF_Q + kmajor_sw128(L::NB, h, u * 8)) = raw;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tO = tmem + 16u;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    constexpr uint32_t ID_S = idesc_bf16_f32(DEC_KS, L::NB, 0, 0);
    constexpr uint32_t ID_O = idesc_bf16_f32(D, L::NB, 0, 1);  // A = V^T, MN-major

    // ---- S^T = K Q^T, issued by warp 0 (converged; one elected lane per operation)
    if (warp == 0) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar_k, 0, abort_flag, lim));
        if (ok) {
            const uint64_t ak = smem_desc_sw128(sbase + L::OFF_K, 16, 1024);
            const uint64_t bq = smem_desc_sw128(sbase + L::OFF_Q, 16, 1024);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t offk = ((k >> 2) * (DEC_KS * 128) + (k & 3) * 32) >> 4;
                const uint32_t offq = ((k >> 2) * (L::NB * 128) + (k & 3) * 32) >> 4;
                mma_ss_elect(tS, ak + offk, bq + offq, ID_S, k > 0 ? 1u : 0u);
            }
            mma_commit_elect(bar_m);
        }
    }
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar_m, 0, abort_flag, lim));
    tc_fence_after();
    uint32_t sr[16];
    if (ok) tmem_ld16(tS + lane_off, sr);  // warp-uniform condition: the load is collective
    const bool valid = ok && t < nk;
    float s[G];
#pragma unroll
    for (int h = 0; h < G; ++h) s[h] = valid ? __uint_as_float(sr[h]) * p.scale_log2 : -INFINITY;

    // ---- per head: maximum and sum over the split (warp shuffles, then the warps)
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float v = s[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) red[warp * G + h] = v;
    }
    __syncthreads();
    float e[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float mh = red[h];
#pragma unroll
        for (int w = 1; w < DEC_WARPS; ++w) mh = fmaxf(mh, red[w * G + h]);
        e[h] = valid ? exp2f(s[h] - mh) : 0.f;
        float v = e[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[DEC_WARPS * G + warp * G + h] = v;
    }
    // the weights of slot t as column t of the B operand P^T (rows h >= G zero)
#pragma unroll
    for (int h = 0; h < L::NB; ++h)
        *reinterpret_cast<__nv_bfloat16*>(smem + L::OFF_P + kmajor_sw128(L::NB, h, t)) =
            __float2bfloat16_rn(h < G ? e[h] : 0.f);
    // slots past the window's end may hold anything, even NaN, and a zero weight does not
    // cancel a NaN in the product: their V rows are zeroed
    if (ok) ok = mbar_wait_bounded(bar_v, 0, abort_flag, lim);
    if (ok && t >= nk) {
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            uint4* row = reinterpret_cast<uint4*>(smem + L::OFF_V + c * (DEC_KS * 128) + t * 128);
#pragma unroll
            for (int u = 0; u < 8; ++u) row[u] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    fence_proxy_async_smem();
    const bool go = __syncthreads_and(ok) != 0;

    // ---- O^T = V^T P^T over the split's 128 slots, issued by warp 0
    if (go && warp == 0) {
        const uint64_t av = smem_desc_sw128(sbase + L::OFF_V, DEC_KS * 128, 1024);
        const uint64_t bp = smem_desc_sw128(sbase + L::OFF_P, 16, 1024);
#pragma unroll
        for (int k = 0; k < DEC_KS / 16; ++k) {
            const uint32_t offv = (k * 2048) >> 4;  // 16 slots = 16 rows of 128 bytes
            const uint32_t offp = ((k >> 2) * (L::NB * 128) + (k & 3) * 32) >> 4;
            mma_ss_elect(tO, av + offv, bp + offp, ID_O, k > 0 ? 1u : 0u);
        }
        mma_commit_elect(bar_m);
    }
    ok = __all_sync(0xffffffffu, go && mbar_wait_bounded(bar_m, 1, abort_flag, lim));
    tc_fence_after();
    if (ok) {
        uint32_t orow[16];
        tmem_ld16(tO + lane_off, orow);  // output column t of every head
        const size_t row0 = ((size_t)b * p.Hq + (size_t)hk * g) * p.nsplit + split;
#pragma unroll
        for (int h = 0; h < G; ++h)
            if (h < g) p.part_o[(row0 + (size_t)h * p.nsplit) * D + t] = __uint_as_float(orow[h]);
        if (t < g) {
            float l = 0.f, mh = -INFINITY;
#pragma unroll
            for (int w = 0; w < DEC_WARPS; ++w) {
                l += red[DEC_WARPS * G + w * G + t];
                mh = fmaxf(mh, red[w * G + t]);
            }
            const size_t row = row0 + (size_t)t * p.nsplit;
            p.part_ml[row * 2] = mh;
            p.part_ml[row * 2 + 1] = l;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
    if (t == 0 && *abort_flag) atomicExch(p.status, 6 /* SWA_ERR_TIMEOUT */);
}

template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const __grid_constant__ DecParams p) {
    const int bh = blockIdx.x;  // b * Hq + h
    const int b = bh / p.Hq;
    const int c = threadIdx.x;
    const int posb = p.pos[b];
    const int nvalid = posb < 0 ? 0 : min(posb + 1, p.W);
    const int ns = (nvalid + DEC_KS - 1) / DEC_KS;
    const float* __restrict__ ml = p.part_ml + (size_t)bh * p.nsplit * 2;
    const float* __restrict__ po = p.part_o + (size_t)bh * p.nsplit * D + c;
    // splits in batches of eight: the loads of a batch are issued together (one after the
    // other they would expose a memory latency per split); the sums keep the split order
    float mx = -INFINITY;
    for (int s0 = 0; s0 < ns; s0 += 8) {
        float mv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mv[u] = (s0 + u < ns) ? __ldg(ml + 2 * (s0 + u)) : -INFINITY;
#pragma unroll
        for (int u = 0; u < 8; ++u) mx = fmaxf(mx, mv[u]);
    }
    float l = 0.f, o = 0.f;
    for (int s0 = 0; s0 < ns; s0 += 8) {
        float mv[8], lv[8], ov[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const bool in = s0 + u < ns;
            mv[u] = in ? __ldg(ml + 2 * (s0 + u)) : 0.f;
            lv[u] = in ? __ldg(ml + 2 * (s0 + u) + 1) : 0.f;
            ov[u] = in ? __ldg(po + (size_t)(s0 + u) * D) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (s0 + u < ns) {
                const float w = exp2f(mv[u] - mx);
                l += lv[u] * w;
                o += ov[u] * w;
            }
        }
    }
    p.out[(size_t)bh * D + c] = __float2bfloat16_rn(l > 0.f ? o / l : 0.f);
}

// Write n new K and V rows per (sequence, KV head) into the rolling caches: row r holds
// position pos + r and goes to slot (pos + r) mod W; of a block longer than W only the last
// W rows are written (the others would be overwritten at once).  grid (rows, up to 65535
// (sequence, KV head) pairs walked with a stride of gridDim.y), D/8 threads (16-byte units).
// The slot is formed in 64-bit arithmetic: pos + r may exceed the int range.
template <int D>
__global__ void __launch_bounds__(D / 8) cache_append_kernel(const __nv_bfloat16* k_new,
                                                             const __nv_bfloat16* v_new,
                                                             __nv_bfloat16* k_cache,
                                                             __nv_bfloat16* v_cache,
                                                             const int* pos, int n_bh, int Hkv,
                                                             int W, int n) {
    const int r = n - min(n, W) + (int)blockIdx.x;
    const int u = threadIdx.x;
    for (int bh = (int)blockIdx.y; bh < n_bh; bh += (int)gridDim.y) {  // b * Hkv + hk
        const int posb = pos[bh / Hkv];
        if (posb < 0) continue;
        const size_t slot = (size_t)(((long long)posb + r) % W);
        const size_t src = ((size_t)bh * n + r) * D;
        reinterpret_cast<uint4*>(k_cache + ((size_t)bh * W + slot) * D)[u] =
            reinterpret_cast<const uint4*>(k_new + src)[u];
        reinterpret_cast<uint4*>(v_cache + ((size_t)bh * W + slot) * D)[u] =
            reinterpret_cast<const uint4*>(v_new + src)[u];
    }
}

// Copy the nctx positions pos0 - nctx .. pos0 - 1 out of the rolling caches, in time order,
// into rows 0 .. nctx-1 of contiguous context buffers [B*Hkv][ctx_rows][D].  grid (rows,
// up to 65535 (sequence, KV head) pairs walked with a stride of gridDim.y).
template <int D>
__global__ void __launch_bounds__(D / 8) cache_gather_kernel(const __nv_bfloat16* k_cache,
                                                             const __nv_bfloat16* v_cache,
                                                             __nv_bfloat16* k_ctx,
                                                             __nv_bfloat16* v_ctx, int n_bh,
                                                             int W, int pos0, int nctx,
                                                             int ctx_rows) {
    const int r = blockIdx.x;
    const size_t slot = (size_t)(((long long)pos0 - nctx + r) % W);
    const int u = threadIdx.x;
    for (int bh = (int)blockIdx.y; bh < n_bh; bh += (int)gridDim.y) {
        const size_t dst = ((size_t)bh * ctx_rows + r) * D;
        reinterpret_cast<uint4*>(k_ctx + dst)[u] =
            reinterpret_cast<const uint4*>(k_cache + ((size_t)bh * W + slot) * D)[u];
        reinterpret_cast<uint4*>(v_ctx + dst)[u] =
            reinterpret_cast<const uint4*>(v_cache + ((size_t)bh * W + slot) * D)[u];
    }
}

}  // namespace swa
