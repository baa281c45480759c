// attn_bwd.cuh -- sm_103a backward pass of causal sliding-window attention: dq, dk, dv.
//
// What it computes ("SWA：滑动窗口注意力与跨层信息传递" §3.1 defines the forward
// out_i = sum_j a_ij v_j, a_ij = softmax_j(scale q_i.k_j + M_ij) over the window
// max(0, i-W+1) <= j <= i; "注意力变体" exercises 2-3 train models with such layers, which
// needs its gradients).  For an upstream gradient dout, by the chain rule through the row
// softmax:
//   dv_j = sum_i a_ij dout_i,        dp_ij = dout_i . v_j,
//   ds_ij = a_ij (dp_ij - delta_i),  delta_i = sum_j a_ij dp_ij = dout_i . out_i,
//   dq_i = scale sum_j ds_ij k_j,    dk_j = scale sum_i ds_ij q_i.
// a_ij is recomputed from the forward's row log-sum-exp: a_ij = exp(scale q_i.k_j - lse_i).
//
// Three kernels, launched in order on one stream:
//   bwd_delta_kernel      delta_i = dout_i . out_i (bf16 in, fp32 out), one row per thread
//   attn_bwd_kernel<D, 0> (dk, dv) one CTA per (batch, KV head, 128-key tile): walks the
//                         query tiles of the group's heads that see the tile; S^T = K Q^T and
//                         dP^T = V dO^T on tcgen05, P^T and dS^T from them, then
//                         dV += P^T dO and dK += dS^T Q accumulate in tensor memory
//   attn_bwd_kernel<D, 1> (dq) one CTA per (batch, query head, 128-row tile): walks the KV
//                         tiles of the row tile's window; S = Q K^T, dP = dO V^T, dS,
//                         dQ += dS K
// The dq kernel recomputes S and dP instead of having the dk/dv kernel scatter dq with
// atomics: dq stays deterministic and no fp32 dq buffer is needed.
//
// CTA organisation (320 threads): warps 0-7 compute; warps w and w + 4 share TMEM lanes
// 32 (w % 4) .. 32 (w % 4) + 31 (a query row each in the dq kernel, a key row each in the
// dk/dv kernel) and split the 128 columns of a step, 64 each, so two warps per lane quarter
// overlap their exponentials; warp 8 lane 0 loads tiles with TMA, warp 9 owns TMEM and
// issues the MMAs (converged warp, one elected lane per operation).  P^T and dS^T (or dS)
// are packed to bf16 pairs over the first 32 of each half's 64 columns, i.e. TMEM columns
// [0, 32) and [64, 96) of the S and dP regions; a warp overwrites only columns it has read.
// A 32-column chunk that no lane of a warp may read is neither loaded nor exponentiated.
// Every MMA form here is one the forward kernel uses: S-type products with both operands
// K-major from shared memory, and accumulating products whose A operand (P or dS, bf16
// packed in pairs) is read from tensor memory and whose B operand is a K-major tile read as
// MN-major.  Every wait is bounded; a timeout raises the CTA's abort flag, every role
// leaves its loop, and the status word reports SWA_ERR_TIMEOUT.
#pragma once

#include "attn_fwd.cuh"

namespace swa {

struct BwdParams {
    CUtensorMap tm_q;   // [B*Hq][N][d] bf16
    CUtensorMap tm_k;   // [B*Hkv][N][d]
    CUtensorMap tm_v;
    CUtensorMap tm_do;  // [B*Hq][N][d]
    const float* lse;   // [B, Hq, N] natural-log row log-sum-exp of the forward
    const float* delta; // [B, Hq, N] dout . out
    __nv_bfloat16* dq;  // [B, Hq, N, d]
    __nv_bfloat16* dk;  // [B, Hkv, N, d]
    __nv_bfloat16* dv;  // [B, Hkv, N, d]
    int* status;
    unsigned long long wait_limit_ns;
    int B, Hq, Hkv, N, W;
    float scale, scale_log2;
};

constexpr int BWD_THREADS = 320;
constexpr int BWD_COMPUTE_WARPS = 8;
constexpr int BWD_PRODUCER_WARP = 8;
constexpr int BWD_MMA_WARP = 9;
constexpr float LOG2E_F = 1.4426950408889634f;

template <int D>
struct BwdLayout {
    static constexpr int TB = BM * D * 2;    // one 128-row bf16 tile (D/64 boxes of 16 KiB)
    static constexpr int OFF_FIX = 0;        // the two tiles the CTA keeps (Q, dO or K, V)
    static constexpr int OFF_RING = 2 * TB;  // two stages, each two tiles
    static constexpr int OFF_BAR = OFF_RING + 4 * TB;
    static constexpr int BAR_FIX = 0;
    static constexpr int BAR_FULL = 1;   // two
    static constexpr int BAR_EMPTY = 3;  // two
    static constexpr int BAR_SP = 5;     // S and dP products of a step are in TMEM
    static constexpr int BAR_DS = 6;     // the step's P / dS are in TMEM (one arrival per warp)
    static constexpr int BAR_FIN = 7;    // every MMA of the CTA has completed
    static constexpr int NBARS = 8;
    static constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM + 4;
    static constexpr int END = OFF_ABORT + 4;
    // at least 116 KiB, so that one CTA holds an SM: each allocates all 512 TMEM columns
    static constexpr int MIN_BYTES = 116 * 1024;
    static constexpr int BYTES = (END + 1024 > MIN_BYTES) ? END + 1024 : MIN_BYTES;
    static_assert(BYTES <= 232448, "shared memory budget");
    static_assert(TB % 1024 == 0, "1024-byte tile alignment");
};

// One 128-row tile of a [mat][N][D] tensor (rows past N are zero-filled by TMA).
template <int D>
__device__ __forceinline__ void bwd_load_tile(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                              int row, int mat) {
#pragma unroll
    for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * (BM * 128), m, bar, c * 64, row, mat);
}

// Columns [32 c0, 32 c0 + D/2) of fp32 from TMEM lane (the calling thread's), times `mul`,
// to the same columns of one bf16 row (the two warps of a lane quarter store one half each).
template <int D>
__device__ __forceinline__ void bwd_store_half_row(uint32_t taddr, float mul,
                                                   __nv_bfloat16* dst, bool valid, int c0) {
#pragma unroll
    for (int cc = 0; cc < D / 64; ++cc) {
        const int c = c0 + cc;
        uint32_t rr[32];
        tmem_ld32(taddr + c * 32, rr);
        if (valid) {
            uint4* o = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
                const int e = v4 * 8;
                o[v4] = make_uint4(
                    pack_bf16x2(__uint_as_float(rr[e + 0]) * mul, __uint_as_float(rr[e + 1]) * mul),
                    pack_bf16x2(__uint_as_float(rr[e + 2]) * mul, __uint_as_float(rr[e + 3]) * mul),
                    pack_bf16x2(__uint_as_float(rr[e + 4]) * mul, __uint_as_float(rr[e + 5]) * mul),
                    pack_bf16x2(__uint_as_float(rr[e + 6]) * mul, __uint_as_float(rr[e + 7]) * mul));
            }
        }
    }
}

// delta_r = dout_r . out_r for every row r of [rows][D] (bf16), fp32 accumulation.
template <int D>
__global__ void bwd_delta_kernel(const __nv_bfloat16* __restrict__ out,
                                 const __nv_bfloat16* __restrict__ dout, float* __restrict__ delta,
                                 long long rows) {
    const long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const uint4* o = reinterpret_cast<const uint4*>(out + r * D);
    const uint4* g = reinterpret_cast<const uint4*>(dout + r * D);
    float acc = 0.f;
#pragma unroll 4
    for (int c = 0; c < D / 8; ++c) {
        const uint4 a = __ldg(o + c), b = __ldg(g + c);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            acc = fmaf(__uint_as_float(av[u] << 16), __uint_as_float(bv[u] << 16), acc);
            acc = fmaf(__uint_as_float(av[u] & 0xFFFF0000u), __uint_as_float(bv[u] & 0xFFFF0000u),
                       acc);
        }
    }
    delta[r] = acc;
}

// The two kernels share their skeleton; KIND 0 is the dk/dv kernel, KIND 1 the dq kernel.
template <int D, int KIND>
__global__ void __launch_bounds__(BWD_THREADS, 1) attn_bwd_kernel(const __grid_constant__ BwdParams p) {
    using L = BwdLayout<D>;
    constexpr bool DKDV = (KIND == 0);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + L::OFF_BAR + 8u * (uint32_t)i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_ABORT);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM);
    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();
    const uint64_t lim = p.wait_limit_ns;
    const int g = p.Hq / p.Hkv;

    // ---- the CTA's tile and its step sequence
    // dk/dv: blockIdx.y = b * Hkv + hk, the 128 keys from t0; step s reads query head
    //   hk*g + s / nq, query tile i_lo + s % nq (the tiles whose rows can see one of the keys).
    // dq: blockIdx.y = b * Hq + h, the 128 rows from t0; step s reads KV tile j_lo + s.
    const int t0 = (int)blockIdx.x * BM;
    const int bz = (int)blockIdx.y;
    int lo_t, nq, n_steps;
    if (DKDV) {
        lo_t = (int)blockIdx.x;
        const int hi = min(p.N - 1, t0 + BN - 1 + p.W - 1) / BM;
        nq = hi - lo_t + 1;
        n_steps = g * nq;
    } else {
        lo_t = max(0, t0 - p.W + 1) / BN;
        const int hi = min(p.N - 1, t0 + BM - 1) / BN;
        nq = hi - lo_t + 1;
        n_steps = nq;
    }
    const int b = DKDV ? bz / p.Hkv : bz / p.Hq;
    const int kvmat = DKDV ? bz : b * p.Hkv + (bz % p.Hq) / g;  // K / V matrix
    auto step_qmat = [&](int s) -> int {  // query-side matrix (Q, dO, lse, delta) of a step
        return DKDV ? b * p.Hq + (bz % p.Hkv) * g + s / nq : bz;
    };
    auto step_tile = [&](int s) -> int { return lo_t + (DKDV ? s % nq : s); };

    // ---- setup
    if (warp == BWD_MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(bar(L::BAR_FIX), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(L::BAR_FULL + s), 1);
            mbar_init(bar(L::BAR_EMPTY + s), 1);
        }
        mbar_init(bar(L::BAR_SP), 1);
        mbar_init(bar(L::BAR_DS), BWD_COMPUTE_WARPS);
        mbar_init(bar(L::BAR_FIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == BWD_PRODUCER_WARP && lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        tma_prefetch_desc(&p.tm_do);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == BWD_PRODUCER_WARP) {
        // ===================================== TMA producer (lane 0)
        if (lane == 0) {
            bool ok = true;
            mbar_arrive_expect_tx(bar(L::BAR_FIX), 2 * L::TB);
            if (DKDV) {
                bwd_load_tile<D>(sbase + L::OFF_FIX, &p.tm_k, bar(L::BAR_FIX), t0, kvmat);
                bwd_load_tile<D>(sbase + L::OFF_FIX + L::TB, &p.tm_v, bar(L::BAR_FIX), t0, kvmat);
            } else {
                bwd_load_tile<D>(sbase + L::OFF_FIX, &p.tm_q, bar(L::BAR_FIX), t0, bz);
                bwd_load_tile<D>(sbase + L::OFF_FIX + L::TB, &p.tm_do, bar(L::BAR_FIX), t0, bz);
            }
            int issued = 0;
            for (int s = 0; s < n_steps && ok; ++s) {
                const int st = s & 1, use = s >> 1;
                if (use > 0)
                    ok = mbar_wait_bounded(bar(L::BAR_EMPTY + st), (uint32_t)(use - 1) & 1u,
                                           abort_flag, lim);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(L::BAR_FULL + st), 2 * L::TB);
                const uint32_t dst = sbase + L::OFF_RING + (uint32_t)st * 2u * L::TB;
                const int row = step_tile(s) * BM;
                if (DKDV) {
                    const int qm = step_qmat(s);
                    bwd_load_tile<D>(dst, &p.tm_q, bar(L::BAR_FULL + st), row, qm);
                    bwd_load_tile<D>(dst + L::TB, &p.tm_do, bar(L::BAR_FULL + st), row, qm);
                } else {
                    bwd_load_tile<D>(dst, &p.tm_k, bar(L::BAR_FULL + st), row, kvmat);
                    bwd_load_tile<D>(dst + L::TB, &p.tm_v, bar(L::BAR_FULL + st), row, kvmat);
                }
                issued = s + 1;
            }
            // drain: every issued copy must have landed before the CTA may exit
            volatile int never = 0;
            (void)mbar_wait_bounded(bar(L::BAR_FIX), 0u, &never, lim);
            for (int s = max(0, issued - 2); s < issued; ++s)
                (void)mbar_wait_bounded(bar(L::BAR_FULL + (s & 1)), (uint32_t)(s >> 1) & 1u,
                                        &never, lim);
        }
        __syncwarp();
    } else if (warp == BWD_MMA_WARP) {
        // ===================================== MMA issuer (converged warp)
        constexpr uint32_t ID_S = idesc_bf16_f32(BM, BN, 0);
        constexpr uint32_t ID_O = idesc_bf16_f32(BM, D, 1);
        const uint32_t tS = tmem_base;          // S (then P over its first 64 columns)
        const uint32_t tDP = tmem_base + 128u;  // dP (then dS over its first 64 columns)
        const uint32_t tA1 = tmem_base + 256u;  // dk/dv: dV;  dq: dQ
        const uint32_t tA2 = tmem_base + 256u + (uint32_t)D;  // dk/dv: dK
        // fixed operands: A of the two S-type products
        const uint64_t fa0 = smem_desc_sw128(sbase + L::OFF_FIX, 16, 1024);
        const uint64_t fa1 = smem_desc_sw128(sbase + L::OFF_FIX + L::TB, 16, 1024);
        auto wait = [&](uint32_t bb, uint32_t parity) -> bool {
            const bool r = mbar_wait_bounded(bb, parity, abort_flag, lim);
            return __all_sync(0xffffffffu, r);
        };
        bool ok = wait(bar(L::BAR_FIX), 0u);
        for (int s = 0; s < n_steps && ok; ++s) {
            const int st = s & 1;
            ok = wait(bar(L::BAR_FULL + st), (uint32_t)(s >> 1) & 1u);
            if (!ok) break;
            tc_fence_after();
            const uint32_t r0 = sbase + L::OFF_RING + (uint32_t)st * 2u * L::TB;  // Q | K tile
            const uint32_t r1 = r0 + L::TB;                                        // dO | V tile
            const uint64_t b0 = smem_desc_sw128(r0, 16, 1024);
            const uint64_t b1 = smem_desc_sw128(r1, 16, 1024);
            // dk/dv: S^T = K Q^T, dP^T = V dO^T.   dq: S = Q K^T, dP = dO V^T.
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t off = ((k >> 2) * (BM * 128) + (k & 3) * 32) >> 4;
                mma_ss_elect(tS, fa0 + off, b0 + off, ID_S, k > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t off = ((k >> 2) * (BM * 128) + (k & 3) * 32) >> 4;
                mma_ss_elect(tDP, fa1 + off, b1 + off, ID_S, k > 0 ? 1u : 0u);
            }
            mma_commit_elect(bar(L::BAR_SP));
            ok = wait(bar(L::BAR_DS), (uint32_t)s & 1u);
            if (!ok) break;
            tc_fence_after();
            // accumulating products: the ring tiles as MN-major B operands (N = d, K = the
            // tile's 128 rows), P / dS from TMEM as A
            const uint64_t m0 = smem_desc_sw128(r0, BN * 128, 1024);
            const uint64_t m1 = smem_desc_sw128(r1, BN * 128, 1024);
#pragma unroll
            for (int k = 0; k < BN / 16; ++k) {
                const uint64_t koff = (uint64_t)((k * 2048) >> 4);
                const uint32_t acc = (s > 0 || k > 0) ? 1u : 0u;
                // packed pairs of k-step k: columns (k / 4) 64 + (k % 4) 8 of S / dP
                const uint32_t pc = (uint32_t)((k >> 2) * 64 + (k & 3) * 8);
                if (DKDV) {
                    mma_ts_elect(tA1, tS + pc, m1 + koff, ID_O, acc);   // dV += P^T dO
                    mma_ts_elect(tA2, tDP + pc, m0 + koff, ID_O, acc);  // dK += dS^T Q
                } else {
                    mma_ts_elect(tA1, tS + pc, m0 + koff, ID_O, acc);   // dQ += dS K
                }
            }
            mma_commit_elect(bar(L::BAR_EMPTY + st));
        }
        // all issued MMAs complete: the compute warps read the accumulators, TMEM may go
        __syncwarp();
        mma_commit_elect(bar(L::BAR_FIN));
        volatile int never = 0;
        (void)mbar_wait_bounded(bar(L::BAR_FIN), 0u, &never, lim);
        __syncwarp();
    } else {
        // ===================================== compute warps (0-7)
        const int quarter = (int)(warp & 3), half = (int)(warp >> 2);
        const int t = quarter * 32 + (int)lane;  // TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem_base + lane_off;
        const uint32_t tDP = tS + 128u;
        const uint32_t tA1 = tS + 256u;
        const uint32_t tA2 = tS + 256u + (uint32_t)D;
        const int my = t0 + t;  // dk/dv: this thread's key;  dq: its query row
        const bool valid = my < p.N;
        const float sl2 = p.scale_log2;
        float lse2_row = 0.f, delta_row = 0.f;  // dq kernel: the row's own values
        if (!DKDV && valid) {
            lse2_row = __ldg(p.lse + (size_t)bz * p.N + my) * LOG2E_F;
            delta_row = __ldg(p.delta + (size_t)bz * p.N + my);
        }
        bool ok = true;
        for (int s = 0; s < n_steps && ok; ++s) {
            // per-column values of the step's query tile (dk/dv): lane l of this warp's chunk
            // cc holds query column 32 (2 half + cc) + l, handed to the other lanes by shuffles
            float lse2_c[2], delta_c[2];
            const int ct = step_tile(s);
            if (DKDV) {
                const size_t base = (size_t)step_qmat(s) * p.N;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int qc = ct * BM + (2 * half + cc) * 32 + (int)lane;
                    lse2_c[cc] = (qc < p.N) ? __ldg(p.lse + base + qc) * LOG2E_F : 0.f;
                    delta_c[cc] = (qc < p.N) ? __ldg(p.delta + base + qc) : 0.f;
                }
            }
            ok = mbar_wait_bounded(bar(L::BAR_SP), (uint32_t)s & 1u, abort_flag, lim);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            // allowed pairs: key j and query i with i - W < j <= i, both < N
            //   dk/dv: this thread's key j = my, column = query ct*128 + col
            //   dq:    this thread's query i = my, column = key ct*128 + col
            int a, bnd;  // allowed columns [a, bnd]
            if (DKDV) {
                const int q0 = ct * BM;
                a = my - q0;                                   // i >= j
                bnd = min(my + p.W - 1, p.N - 1) - q0;         // i <= j + W - 1, i < N
                if (!valid) bnd = -1;
            } else {
                const int k0 = ct * BN;
                a = max(0, my - p.W + 1) - k0;
                bnd = my - k0;
                if (!valid) bnd = -1;
            }
            // the warp's allowed columns lie in [wa, wb]
            int la = max(a, 0), lb = min(bnd, BN - 1);
            if (la > lb) {
                la = BN;
                lb = -1;
            }
            const int wa = __reduce_min_sync(0xffffffffu, la);
            const int wb = __reduce_max_sync(0xffffffffu, lb);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * half + cc;
                uint32_t pk[16], dk16[16];
                if (c * 32 <= wb && c * 32 + 31 >= wa) {  // warp-uniform
                    uint32_t sr[32], dr[32];
                    tmem_ld32(tS + c * 32, sr);
                    tmem_ld32(tDP + c * 32, dr);
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        float pv[2], dsv[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int col = c * 32 + 2 * u + e;
                            float l2, dl;
                            if (DKDV) {
                                l2 = __shfl_sync(0xffffffffu, lse2_c[cc], 2 * u + e);
                                dl = __shfl_sync(0xffffffffu, delta_c[cc], 2 * u + e);
                            } else {
                                l2 = lse2_row;
                                dl = delta_row;
                            }
                            const bool in = (col >= a) && (col <= bnd);
                            pv[e] = in ? fast_exp2(fmaf(__uint_as_float(sr[2 * u + e]), sl2, -l2))
                                       : 0.f;
                            dsv[e] = pv[e] * (__uint_as_float(dr[2 * u + e]) - dl);
                        }
                        pk[u] = pack_bf16x2(pv[0], pv[1]);
                        dk16[u] = pack_bf16x2(dsv[0], dsv[1]);
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u) pk[u] = dk16[u] = 0u;
                }
                // packed columns: 64 half + 16 cc .. + 16, inside the half's first chunk, which
                // this warp has already read
                const uint32_t pc = (uint32_t)(half * 64 + cc * 16);
                if (DKDV) {
                    tmem_st16(tS + pc, pk);     // P^T over S^T
                    tmem_st16(tDP + pc, dk16);  // dS^T over dP^T
                } else {
                    tmem_st16(tS + pc, dk16);   // dS over S
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::BAR_DS));
        }
        if (ok) {
            ok = mbar_wait_bounded(bar(L::BAR_FIN), 0u, abort_flag, lim);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
            const size_t row = (size_t)bz * p.N + (size_t)(valid ? my : 0);
            const int c0 = half * (D / 64);
            if (DKDV) {
                bwd_store_half_row<D>(tA1, 1.f, p.dv + row * D, valid, c0);
                bwd_store_half_row<D>(tA2, p.scale, p.dk + row * D, valid, c0);
            } else {
                bwd_store_half_row<D>(tA1, p.scale, p.dq + row * D, valid, c0);
            }
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == BWD_MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicExch(p.status, 6 /* SWA_ERR_TIMEOUT */);
}

}  // namespace swa
