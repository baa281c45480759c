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
// CTA organisation (576 threads): warps 0-15 compute; warps w, w + 4, w + 8, w + 12 share
// TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31 (a query row each in the dq kernel, a key row each
// in the dk/dv kernel) and split the 128 columns of a step, 32 each, so four warps per lane
// quarter overlap their latencies; warp 16 lane 0 loads tiles with TMA, warp 17 owns TMEM and
// issues the MMAs (converged warp, one elected lane per operation).  P^T (dk/dv) and dS
// (dq) are packed to bf16 pairs over the first 16 of each warp's 32 columns of their S
// region; a warp overwrites only columns it has read.  dS^T (dk/dv) goes to a 128 x 128 shared-memory tile in the 128-byte-swizzled
// K-major layout, the A operand of dK += dS^T Q.
// Every MMA form here is one the forward kernel uses: S-type products with both operands
// K-major from shared memory, accumulating products whose A operand (P^T or dS, bf16 packed
// in pairs) is read from tensor memory or (dS^T) from shared memory and whose B operand is a
// K-major tile read as MN-major.  Every wait is bounded; a timeout raises the CTA's abort
// flag, every role leaves its loop, and the status word reports SWA_ERR_TIMEOUT.
#pragma once

#include "attn_fwd.cuh"

namespace swa {

struct BwdParams {
    CUtensorMap tm_q;   // [B*Hq][N][d] bf16
    CUtensorMap tm_k;   // [B*Hkv][N][d]
    CUtensorMap tm_v;
    CUtensorMap tm_do;  // [B*Hq][N][d]
    CUtensorMap tm_k2;  // strided / global prefix: compact keys, row r = key r * stride
    CUtensorMap tm_v2;  // the same rows of V
    const float* lse;   // [B, Hq, N] natural-log row log-sum-exp of the forward
    const float* delta; // [B, Hq, N] dout . out
    __nv_bfloat16* dq;  // [B, Hq, N, d]
    __nv_bfloat16* dk;  // [B, Hkv, N, d]
    __nv_bfloat16* dv;  // [B, Hkv, N, d]
    float* cpart;       // compact keys: [2][cchunks][B*Hkv][ncomp_pad][d] fp32 partial dK, dV
    int* status;
    unsigned long long wait_limit_ns;
    int B, Hq, Hkv, N, W;
    // local + strided and window + global prefix: row i also reads the compact keys r * stride
    // with r < ncomp(i) = min(ceil(lo(i) / stride), cap), lo(i) = max(0, i - W + 1) (the keys
    // before its window); cap = 0 is the plain window
    int stride, cap;
    int ncomp;          // compact keys any row reads: ncomp(N - 1)
    int ncomp_pad;      // ncomp rounded up to a whole 128-row tile
    int cchunks;        // query-tile chunks of the compact dk/dv pass
    // the second map of differential attention enters the loss with weight mu_h = -lambda_h:
    // mu_mode 1 scales the weights in dV and the dS of every step by mu of its query head
    int mu_mode;
    float lam;                // lambda of every head, unless lam_heads is set
    const float* lam_heads;   // [Hq] per-head lambda (device), or null
    float* dv32_out;          // dk/dv: write dV unrounded (fp32 [B*Hkv][N][d]) here, not dv
    const float* dv32_in;     // dk/dv: fp32 [B*Hkv][N][d] added to dV before rounding, or null
    float scale, scale_log2;
};

#ifndef SWA_BWD_COMPUTE_WARPS
#define SWA_BWD_COMPUTE_WARPS 16
#endif
// compute warps: four per TMEM lane quarter, each taking BWD_CW of a step's 128 columns
constexpr int BWD_COMPUTE_WARPS = SWA_BWD_COMPUTE_WARPS;
constexpr int BWD_CW = 128 / (BWD_COMPUTE_WARPS / 4);
constexpr int BWD_NCH = BWD_CW / 32;  // 32-column chunks per warp and step
constexpr int BWD_PRODUCER_WARP = BWD_COMPUTE_WARPS;
constexpr int BWD_MMA_WARP = BWD_COMPUTE_WARPS + 1;
constexpr int BWD_THREADS = 32 * (BWD_COMPUTE_WARPS + 2);
static_assert(BWD_CW == 32 || BWD_CW == 64, "8 or 16 compute warps");
constexpr float LOG2E_F = 1.4426950408889634f;

template <int D, int KIND>
struct BwdLayout {
    static constexpr int TB = BM * D * 2;    // one 128-row bf16 tile (D/64 boxes of 16 KiB)
    // The moving tiles come through two rings, so each is freed as soon as its last product
    // is done.  Ring A holds the B operand of S (dk/dv: Q, read again by dK; dq: K, read again
    // by dQ); ring B that of dP (dk/dv: dO, read again by dV; dq: V).  Ring A has three
    // entries, so the next step's tile is in place when S(s+1) is issued; at d = 64 ring B
    // has three as well (the tiles are half the size).
    static constexpr int NA = 3;
    static constexpr int NB = (D == 128) ? 2 : 3;
    static constexpr int OFF_FIX = 0;        // the two tiles the CTA keeps (K, V or Q, dO)
    static constexpr int OFF_RA = 2 * TB;
    static constexpr int OFF_RB = OFF_RA + NA * TB;
    static constexpr int OFF_DS = OFF_RB + NB * TB;
    // d = 64 dk/dv kinds: each compute warp's query columns of lse2 and delta, read as
    // broadcasts instead of warp shuffles (at d = 128 they would displace a ring entry, and
    // measured no faster)
    static constexpr bool LSE_SMEM = (KIND == 0) && (D == 64);
    static constexpr int OFF_LSE = OFF_DS;
    static constexpr int LSE_BYTES = LSE_SMEM ? BWD_COMPUTE_WARPS * 2 * BWD_CW * 4 : 0;
    static constexpr int OFF_BAR = OFF_LSE + LSE_BYTES;
    static constexpr int BAR_FIX = 0;
    static constexpr int BAR_AFULL = 1;    // three (ring A entries)
    static constexpr int BAR_AEMPTY = 4;   // three
    static constexpr int BAR_BFULL = 7;    // three (ring B entries)
    static constexpr int BAR_BEMPTY = 10;  // three
    static constexpr int BAR_SREADY = 13;  // S is in TMEM
    static constexpr int BAR_DPREADY = 15; // dP is in TMEM
    static constexpr int BAR_P = 16;       // dk/dv: P^T is in TMEM (one arrival per warp)
    static constexpr int BAR_SFREE = 17;   // dq: S has been read (one arrival per warp)
    static constexpr int BAR_DS = 18;      // dS^T / dS is in TMEM, packed over dP
    static constexpr int BAR_QT = 19;      // dq: Q and dO are in TMEM (one arrival per warp)
    static constexpr int BAR_FIN = 21;     // every MMA of the CTA has completed
    static constexpr int NBARS = 22;
    static constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM + 4;
    static constexpr int END = OFF_ABORT + 4;
    // at least 116 KiB, so that one CTA holds an SM: each allocates all 512 TMEM columns
    static constexpr int MIN_BYTES = 116 * 1024;
    static constexpr int BYTES = (END + 1024 > MIN_BYTES) ? END + 1024 : MIN_BYTES;
    static_assert(BYTES <= 232448, "shared memory budget");
    static_assert(TB % 1024 == 0 && OFF_DS % 1024 == 0, "1024-byte tile alignment");
};

// One 128-row tile of a [mat][N][D] tensor (rows past N are zero-filled by TMA).
template <int D>
__device__ __forceinline__ void bwd_load_tile(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                              int row, int mat) {
#pragma unroll
    for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * (BM * 128), m, bar, c * 64, row, mat);
}

template <int CH>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[CH]) {
    if constexpr (CH == 32)
        tmem_ld32(taddr, r);
    else
        tmem_ld16(taddr, r);
}

// Columns [col0, col0 + NC) of fp32 from TMEM lane (the calling thread's), times `mul`, to
// the same columns of one bf16 row (the warps of a lane quarter store one share each).
// `extra` (or null): n fp32 rows, `stride` floats apart, added to the columns before `mul`.
template <int NC>
__device__ __forceinline__ void bwd_store_cols(uint32_t taddr, float mul, __nv_bfloat16* dst,
                                               bool valid, int col0,
                                               const float* extra = nullptr, int n = 0,
                                               size_t stride = 0) {
    constexpr int CH = NC < 32 ? NC : 32;
#pragma unroll
    for (int cc = 0; cc < NC / CH; ++cc) {
        const int c = col0 + cc * CH;
        uint32_t rr[CH];
        tmem_ld_cols<CH>(taddr + c, rr);
        if (valid && extra != nullptr) {
            for (int i = 0; i < n; ++i) {
                const float* x = extra + (size_t)i * stride + c;
#pragma unroll
                for (int e = 0; e < CH; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) + x[e]);
            }
        }
        if (valid) {
            uint4* o = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int v4 = 0; v4 < CH / 8; ++v4) {
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

// Columns [col0, col0 + NC) of fp32 from TMEM lane to the same columns of an fp32 row (zeros
// when `have` is false: no product wrote the accumulator).  `have` must be the same in every
// lane of the warp (tcgen05.ld is warp-collective); only lanes with `valid` store.
template <int NC>
__device__ __forceinline__ void bwd_store_cols_f32(uint32_t taddr, float* dst, bool have,
                                                   bool valid, int col0) {
    constexpr int CH = NC < 32 ? NC : 32;
#pragma unroll
    for (int cc = 0; cc < NC / CH; ++cc) {
        const int c = col0 + cc * CH;
        uint32_t rr[CH];
        if (have) {
            tmem_ld_cols<CH>(taddr + c, rr);
        } else {
#pragma unroll
            for (int e = 0; e < CH; ++e) rr[e] = 0u;
        }
        if (!valid) continue;
        float4* o = reinterpret_cast<float4*>(dst + c);
#pragma unroll
        for (int v4 = 0; v4 < CH / 4; ++v4)
            o[v4] = make_float4(__uint_as_float(rr[4 * v4]), __uint_as_float(rr[4 * v4 + 1]),
                                __uint_as_float(rr[4 * v4 + 2]), __uint_as_float(rr[4 * v4 + 3]));
    }
}

// The weight mu of query head h (1, or -lambda_h for the second differential map), as the
// log2 of its magnitude (folded into the row's log-sum-exp: |mu| p = exp2(x - lse2 + log2|mu|))
// and the sign bits to flip in a packed bf16 pair.
__device__ __forceinline__ void bwd_mu(const BwdParams& p, int h, float& log2_abs,
                                       uint32_t& sign2) {
    log2_abs = 0.f;
    sign2 = 0u;
    if (p.mu_mode) {
        const float mu = -(p.lam_heads ? p.lam_heads[h] : p.lam);
        log2_abs = log2f(fabsf(mu));  // -inf for mu = 0: every weight becomes 0
        sign2 = signbit(mu) ? 0x80008000u : 0u;
    }
}

// compact keys row i reads: the multiples of the stride before its window start, at most cap
__device__ __forceinline__ int bwd_ncomp(const BwdParams& p, int i) {
    const int lo = max(0, i - p.W + 1);
    return min((lo + p.stride - 1) / p.stride, p.cap);
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

// Sum the compact pass's cchunks partial sums into the first: part[i] += part[c * slot + i]
// for c = 1 .. cchunks-1, for the dk and the dv halves (2 * slot floats in all), so the window
// dk/dv kernel adds one row per compact key.  A fixed order: deterministic.
__global__ void __launch_bounds__(256) bwd_compact_reduce_kernel(float* __restrict__ part,
                                                                 int cchunks, long long slot) {
    const long long n = 2 * slot;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const long long half = i / slot, j = i % slot;
        float* base = part + half * (long long)cchunks * slot;
        float acc = base[j];
        for (int c = 1; c < cchunks; ++c) acc += base[(long long)c * slot + j];
        base[j] = acc;
    }
}

// dlam[h] = -sum over batches and rows of delta[b, h, i] (the gradient of a differential
// head's lambda: d out_i / d lambda = -(A2 V)_i, and delta2_i = dout_i . (A2 V)_i); one CTA of
// 256 threads per head, a fixed summation order, so the result is deterministic.
__global__ void __launch_bounds__(256) bwd_dlam_kernel(const float* __restrict__ delta2,
                                                       float* __restrict__ dlam, int B, int Hq,
                                                       int N) {
    __shared__ float part[256];
    const int h = blockIdx.x;
    float acc = 0.f;
    for (int b = 0; b < B; ++b) {
        const float* r = delta2 + ((size_t)b * Hq + h) * N;
        for (int i = threadIdx.x; i < N; i += 256) acc += r[i];
    }
    part[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) dlam[h] = -part[0];
}

// The kernels share their set-up; KIND 0 is the dk/dv kernel, KIND 1 the dq kernel, KIND 2
// the dk/dv kernel of the compact keys (local + strided and global-prefix masks: a compact key
// r, at position r * stride, is read by every row i >= r * stride + W; the kernel walks those
// rows in chunks and writes fp32 partial sums that the KIND 0 kernel adds before rounding).
// In those masks the dq kernel walks the row tile's compact tiles before its window tiles.
//
// Pipelining.  A step's products are issued so that the tensor core works on one step while
// the compute warps work on another, and each ring entry is released by its last product.
//   dk/dv: per step s the issuer waits for P^T(s) (packed over S^T in TMEM) and issues
//          dV += P^T(s) dO(s), then S^T(s+1) (after dV(s) in issue order, so it cannot
//          overwrite P^T(s) too early); once dS^T(s) is packed over dP^T(s) in TMEM it
//          issues dK += dS^T(s) Q(s) and then dP^T(s+1), which overwrites dS^T(s) only after
//          dK(s) in issue order.  The compute warps form dS^T(s) while dV(s) and S^T(s+1)
//          run, and P^T(s+1) while dK(s) and dP^T(s+1) run.  With both A operands of the
//          accumulating products in TMEM, a step reads 64 KiB less of shared memory, whose
//          128 bytes per cycle the S-type products (both operands from shared memory) and the
//          TMA fills otherwise nearly exhaust.
//   dq:    S has two TMEM regions, so S(s+1) is issued at the start of step s; dP(s+1)
//          once dP(s) has been read; dQ += dS(s) K(s) once dS(s) (packed over S(s)) is in.
// Every barrier completes at most one phase ahead of its waiters: each next phase needs an
// event that follows the waiter's previous wait (the per-region barriers of the dq kernel
// exist for exactly this).
template <int D, int KIND>
__global__ void __launch_bounds__(BWD_THREADS, 1) attn_bwd_kernel(const __grid_constant__ BwdParams p) {
    using L = BwdLayout<D, KIND == 1 ? 1 : 0>;
    constexpr bool DKDV = (KIND != 1);
    constexpr bool COMPACT = (KIND == 2);
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
    // compact: blockIdx.x = compact tile * cchunks + chunk; t0 is a compact row (key r)
    const int ctile = COMPACT ? (int)blockIdx.x / p.cchunks : 0;
    const int chunk = COMPACT ? (int)blockIdx.x % p.cchunks : 0;
    const int t0 = (COMPACT ? ctile : (int)blockIdx.x) * BM;
    const int bz = (int)blockIdx.y;
    const int n_qtiles = (p.N + BM - 1) / BM;
    int lo_t, nq, n_steps, n_ct = 0;  // n_ct: dq kernel, compact tiles before the window's
    if (KIND == 0) {
        lo_t = (int)blockIdx.x;
        const int hi = min(p.N - 1, t0 + BN - 1 + p.W - 1) / BM;
        nq = hi - lo_t + 1;
        n_steps = g * nq;
    } else if (COMPACT) {
        // rows from the first reader of the tile's first key, in cchunks equal ranges
        const long long r_first = (long long)t0 * p.stride + p.W;
        const int qt0 = (t0 < p.ncomp && r_first < p.N) ? (int)(r_first / BM) : n_qtiles;
        const int per = (n_qtiles - qt0 + p.cchunks - 1) / p.cchunks;
        lo_t = qt0 + chunk * per;
        nq = max(0, min(per, n_qtiles - lo_t));
        n_steps = g * nq;
    } else {
        lo_t = max(0, t0 - p.W + 1) / BN;
        const int hi = min(p.N - 1, t0 + BM - 1) / BN;
        nq = hi - lo_t + 1;
        if (p.cap > 0) n_ct = (bwd_ncomp(p, min(p.N - 1, t0 + BM - 1)) + BN - 1) / BN;
        n_steps = n_ct + nq;
    }
    const int b = DKDV ? bz / p.Hkv : bz / p.Hq;
    const int kvmat = DKDV ? bz : b * p.Hkv + (bz % p.Hq) / g;  // K / V matrix
    auto step_qmat = [&](int s) -> int {  // query-side matrix (Q, dO, lse, delta) of a step
        return DKDV ? b * p.Hq + (bz % p.Hkv) * g + s / nq : bz;
    };
    // query tile (dk/dv kinds) or window KV tile (dq) of a step; dq: -1 - c for compact tile c
    auto step_tile = [&](int s) -> int {
        if (DKDV) return lo_t + s % nq;
        return s < n_ct ? -1 - s : lo_t + (s - n_ct);
    };

    // ---- setup
    if (warp == BWD_MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(bar(L::BAR_FIX), 1);
        for (int i = 0; i < 3; ++i) {
            mbar_init(bar(L::BAR_AFULL + i), 1);
            mbar_init(bar(L::BAR_AEMPTY + i), 1);
        }
        for (int i = 0; i < 3; ++i) {
            mbar_init(bar(L::BAR_BFULL + i), 1);
            mbar_init(bar(L::BAR_BEMPTY + i), 1);
        }
        mbar_init(bar(L::BAR_SREADY), 1);
        mbar_init(bar(L::BAR_DS), BWD_COMPUTE_WARPS);
        mbar_init(bar(L::BAR_DPREADY), 1);
        mbar_init(bar(L::BAR_P), BWD_COMPUTE_WARPS);
        mbar_init(bar(L::BAR_SFREE), BWD_COMPUTE_WARPS);
        mbar_init(bar(L::BAR_QT), BWD_COMPUTE_WARPS);
        mbar_init(bar(L::BAR_FIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == BWD_PRODUCER_WARP && lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        tma_prefetch_desc(&p.tm_do);
        if (p.cap > 0) {
            tma_prefetch_desc(&p.tm_k2);
            tma_prefetch_desc(&p.tm_v2);
        }
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
                const CUtensorMap* mk = COMPACT ? &p.tm_k2 : &p.tm_k;
                const CUtensorMap* mv = COMPACT ? &p.tm_v2 : &p.tm_v;
                bwd_load_tile<D>(sbase + L::OFF_FIX, mk, bar(L::BAR_FIX), t0, kvmat);
                bwd_load_tile<D>(sbase + L::OFF_FIX + L::TB, mv, bar(L::BAR_FIX), t0, kvmat);
            } else {
                bwd_load_tile<D>(sbase + L::OFF_FIX, &p.tm_q, bar(L::BAR_FIX), t0, bz);
                bwd_load_tile<D>(sbase + L::OFF_FIX + L::TB, &p.tm_do, bar(L::BAR_FIX), t0, bz);
            }
            // per step: the tile of each ring, the one whose entry frees first (dk/dv: dO;
            // dq: K) first
            auto load_a = [&](int s) -> bool {
                const int e = s % L::NA, use = s / L::NA;
                if (use > 0 && !mbar_wait_bounded(bar(L::BAR_AEMPTY + e), (uint32_t)(use - 1) & 1u,
                                                  abort_flag, lim))
                    return false;
                mbar_arrive_expect_tx(bar(L::BAR_AFULL + e), L::TB);
                const uint32_t dst = sbase + L::OFF_RA + (uint32_t)e * L::TB;
                const int tl = step_tile(s);
                if (DKDV)
                    bwd_load_tile<D>(dst, &p.tm_q, bar(L::BAR_AFULL + e), tl * BM, step_qmat(s));
                else if (tl < 0)  // compact tile -1 - tl
                    bwd_load_tile<D>(dst, &p.tm_k2, bar(L::BAR_AFULL + e), (-1 - tl) * BN, kvmat);
                else
                    bwd_load_tile<D>(dst, &p.tm_k, bar(L::BAR_AFULL + e), tl * BN, kvmat);
                return true;
            };
            auto load_b = [&](int s) -> bool {
                const int e = s % L::NB, use = s / L::NB;
                if (use > 0 && !mbar_wait_bounded(bar(L::BAR_BEMPTY + e), (uint32_t)(use - 1) & 1u,
                                                  abort_flag, lim))
                    return false;
                mbar_arrive_expect_tx(bar(L::BAR_BFULL + e), L::TB);
                const uint32_t dst = sbase + L::OFF_RB + (uint32_t)e * L::TB;
                const int tl = step_tile(s);
                if (DKDV)
                    bwd_load_tile<D>(dst, &p.tm_do, bar(L::BAR_BFULL + e), tl * BM, step_qmat(s));
                else if (tl < 0)
                    bwd_load_tile<D>(dst, &p.tm_v2, bar(L::BAR_BFULL + e), (-1 - tl) * BN, kvmat);
                else
                    bwd_load_tile<D>(dst, &p.tm_v, bar(L::BAR_BFULL + e), tl * BN, kvmat);
                return true;
            };
            int issued_a = 0, issued_b = 0;
            for (int s = 0; s < n_steps && ok; ++s) {
                if (DKDV) {
                    ok = load_b(s);
                    if (ok) issued_b = s + 1;
                    if (ok) ok = load_a(s);
                    if (ok) issued_a = s + 1;
                } else {
                    ok = load_a(s);
                    if (ok) issued_a = s + 1;
                    if (ok) ok = load_b(s);
                    if (ok) issued_b = s + 1;
                }
            }
            // drain: every issued copy must have landed before the CTA may exit
            volatile int never = 0;
            (void)mbar_wait_bounded(bar(L::BAR_FIX), 0u, &never, lim);
            for (int s = max(0, issued_a - L::NA); s < issued_a; ++s)
                (void)mbar_wait_bounded(bar(L::BAR_AFULL + s % L::NA), (uint32_t)(s / L::NA) & 1u,
                                        &never, lim);
            for (int s = max(0, issued_b - L::NB); s < issued_b; ++s)
                (void)mbar_wait_bounded(bar(L::BAR_BFULL + s % L::NB), (uint32_t)(s / L::NB) & 1u,
                                        &never, lim);
        }
        __syncwarp();
    } else if (warp == BWD_MMA_WARP) {
        // ===================================== MMA issuer (converged warp)
        constexpr uint32_t ID_S = idesc_bf16_f32(BM, BN, 0);
        constexpr uint32_t ID_O = idesc_bf16_f32(BM, D, 1);
        // TMEM.  dk/dv: S^T [0,128) (P^T packed over it), dP^T [128,256) (dS^T packed over
        //               it), dV [256,256+D), dK [256+D,256+2D).
        //        dq:    S [0,128), dP [128,256) (dS packed over it), dQ [256,256+D), and the
        //               A operands of S and dP: Q and dO packed in pairs, D/2 columns each.
        const uint32_t tDP = tmem_base + 128u;
        const uint32_t tA1 = tmem_base + 256u;                // dk/dv: dV;  dq: dQ
        const uint32_t tA2 = tmem_base + 256u + (uint32_t)D;  // dk/dv: dK;  dq: Q, then dO
        // fixed operands: A of the two S-type products
        const uint64_t fa0 = smem_desc_sw128(sbase + L::OFF_FIX, 16, 1024);
        const uint64_t fa1 = smem_desc_sw128(sbase + L::OFF_FIX + L::TB, 16, 1024);
        auto wait = [&](uint32_t bb, uint32_t parity) -> bool {
            const bool r = mbar_wait_bounded(bb, parity, abort_flag, lim);
            return __all_sync(0xffffffffu, r);
        };
        auto ring_a = [&](int s) -> uint32_t { return sbase + L::OFF_RA + (uint32_t)(s % L::NA) * L::TB; };
        auto ring_b = [&](int s) -> uint32_t { return sbase + L::OFF_RB + (uint32_t)(s % L::NB) * L::TB; };
        auto wait_a = [&](int s) { return wait(bar(L::BAR_AFULL + s % L::NA), (uint32_t)(s / L::NA) & 1u); };
        auto wait_b = [&](int s) { return wait(bar(L::BAR_BFULL + s % L::NB), (uint32_t)(s / L::NB) & 1u); };
        // an S-type product: D(tmem) = fixed tile (A, K-major) times ring tile (B, K-major);
        // dq: the fixed tile's copy in TMEM (ta, D/2 packed columns) is the A operand
        auto issue_sprod = [&](uint32_t dst, uint64_t fa, uint32_t ta, uint32_t tile) {
            const uint64_t bd = smem_desc_sw128(tile, 16, 1024);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t off = ((k >> 2) * (BM * 128) + (k & 3) * 32) >> 4;
                if (DKDV)
                    mma_ss_elect(dst, fa + off, bd + off, ID_S, k > 0 ? 1u : 0u);
                else
                    mma_ts_elect(dst, ta + (uint32_t)(k * 8), bd + off, ID_S, k > 0 ? 1u : 0u);
            }
        };
        const uint32_t tQ = tA2, tDO = tA2 + (uint32_t)(D / 2);  // dq
        // a ring tile as the MN-major B operand (N = d, K = the tile's 128 rows) of k-step k
        auto mn_b = [&](uint32_t tile, int k) -> uint64_t {
            return smem_desc_sw128(tile, BN * 128, 1024) + (uint64_t)((k * 2048) >> 4);
        };
        // packed pairs of k-step k of P^T / dS in TMEM: each compute warp packs its BWD_CW
        // columns over the first half of them
        auto pcol = [](int k) -> uint32_t {
            return (uint32_t)((k / (BWD_CW / 16)) * BWD_CW + (k % (BWD_CW / 16)) * 8);
        };
        bool ok = wait(bar(L::BAR_FIX), 0u);
        if (ok && !DKDV) ok = wait(bar(L::BAR_QT), 0u);  // dq: Q and dO copied into TMEM
        if (ok && n_steps > 0) ok = wait_a(0);
        if (ok && n_steps > 0) {
            tc_fence_after();
            issue_sprod(tmem_base, fa0, tQ, ring_a(0));  // S(0)
            mma_commit_elect(bar(L::BAR_SREADY));
            ok = wait_b(0);
            if (ok) {
                tc_fence_after();
                issue_sprod(tDP, fa1, tDO, ring_b(0));  // dP(0)
                mma_commit_elect(bar(L::BAR_DPREADY));
                if (!DKDV) mma_commit_elect(bar(L::BAR_BEMPTY));  // dq: V(0) read
            }
        }
        for (int s = 0; s < n_steps && ok; ++s) {
            const bool more = s + 1 < n_steps;
            if (DKDV) {
                ok = wait(bar(L::BAR_P), (uint32_t)s & 1u);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)  // dV += P^T dO
                    mma_ts_elect(tA1, tmem_base + pcol(k), mn_b(ring_b(s), k), ID_O,
                                 (s > 0 || k > 0) ? 1u : 0u);
                mma_commit_elect(bar(L::BAR_BEMPTY + s % L::NB));  // dO(s) read
                if (more) {
                    // S^T(s+1), after dV(s) in issue order (it overwrites P^T(s))
                    ok = wait_a(s + 1);
                    if (!ok) break;
                    tc_fence_after();
                    issue_sprod(tmem_base, fa0, 0u, ring_a(s + 1));
                    mma_commit_elect(bar(L::BAR_SREADY));
                }
                // dK += dS^T Q, dS^T packed over the columns of dP^T(s)
                ok = wait(bar(L::BAR_DS), (uint32_t)s & 1u);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    mma_ts_elect(tA2, tDP + pcol(k), mn_b(ring_a(s), k), ID_O,
                                 (s > 0 || k > 0) ? 1u : 0u);
                mma_commit_elect(bar(L::BAR_AEMPTY + s % L::NA));  // Q(s) read
                if (more) {
                    // dP^T(s+1), after dK(s) in issue order (it overwrites dS^T(s)); the
                    // compute warps read dP^T(s) before they wrote dS^T(s)
                    ok = wait_b(s + 1);
                    if (!ok) break;
                    tc_fence_after();
                    issue_sprod(tDP, fa1, 0u, ring_b(s + 1));
                    mma_commit_elect(bar(L::BAR_DPREADY));
                }
                continue;
            }
            // dq: S(s+1) once the compute warps have read S(s) (its weights stay in their
            // registers); dQ += dS(s) K(s) once dS(s) is packed over dP(s); then dP(s+1),
            // which overwrites dS(s) only after dQ(s) in issue order
            if (more) {
                ok = wait(bar(L::BAR_SFREE), (uint32_t)s & 1u);
                if (ok) ok = wait_a(s + 1);
                if (!ok) break;
                tc_fence_after();
                issue_sprod(tmem_base, fa0, tQ, ring_a(s + 1));
                mma_commit_elect(bar(L::BAR_SREADY));
            }
            ok = wait(bar(L::BAR_DS), (uint32_t)s & 1u);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < BN / 16; ++k)  // dQ += dS K
                mma_ts_elect(tA1, tDP + pcol(k), mn_b(ring_a(s), k), ID_O,
                             (s > 0 || k > 0) ? 1u : 0u);
            mma_commit_elect(bar(L::BAR_AEMPTY + s % L::NA));  // K(s) read
            if (more) {
                ok = wait_b(s + 1);
                if (!ok) break;
                tc_fence_after();
                issue_sprod(tDP, fa1, tDO, ring_b(s + 1));
                mma_commit_elect(bar(L::BAR_DPREADY));
                mma_commit_elect(bar(L::BAR_BEMPTY + (s + 1) % L::NB));  // V(s+1) read
            }
        }
        // all issued MMAs complete: the compute warps read the accumulators, TMEM may go
        __syncwarp();
        mma_commit_elect(bar(L::BAR_FIN));
        volatile int never = 0;
        (void)mbar_wait_bounded(bar(L::BAR_FIN), 0u, &never, lim);
        __syncwarp();
    } else {
        // ===================================== compute warps
        const int quarter = (int)(warp & 3), part = (int)(warp >> 2);
        const int cb = part * BWD_CW;  // this warp's first column of a step
        const int t = quarter * 32 + (int)lane;  // TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tL = tmem_base + lane_off;
        const uint32_t tDP = tL + 128u;
        const uint32_t tA1 = tL + 256u;
        const uint32_t tA2 = tL + 256u + (uint32_t)D;
        const int my = t0 + t;  // dk/dv: this thread's key (compact: key index r);  dq: its row
        const bool valid = COMPACT ? (my < p.ncomp_pad) : (my < p.N);
        const float sl2 = p.scale_log2;
        float lse2_row = 0.f, delta_row = 0.f;  // dq kernel: the row's own values
        float mu_l2 = 0.f;                       // log2 |mu| of the step's query head
        uint32_t mu_sign = 0u;                   // its sign, on a packed bf16 pair
        if (!DKDV) {
            bwd_mu(p, bz % p.Hq, mu_l2, mu_sign);
            if (valid) {
                lse2_row = __ldg(p.lse + (size_t)bz * p.N + my) * LOG2E_F - mu_l2;
                delta_row = __ldg(p.delta + (size_t)bz * p.N + my);
            }
        }
        auto wait = [&](uint32_t bb, uint32_t parity) -> bool {
            const bool r = mbar_wait_bounded(bb, parity, abort_flag, lim);
            return __all_sync(0xffffffffu, r);
        };
        bool ok = true;
        if (!DKDV) {
            // dq: this thread's rows of Q and dO into TMEM, bf16 packed in pairs (the A operands
            // of S and dP): the D packed columns of both are split among the lane quarter's four
            // warps, 16-column pieces read from the swizzled tiles (unit u of row t at u ^ (t & 7))
            ok = wait(bar(L::BAR_FIX), 0u);
            if (ok) {
#pragma unroll
                for (int piece = 0; piece < D / 64; ++piece) {
                    const int gc = part * (D / 4) + piece * 16;  // packed column over Q then dO
                    const int tile = gc / (D / 2), pc = gc % (D / 2);
                    const int e0 = 2 * pc;                       // first element of the piece
                    const uint8_t* row = smem + L::OFF_FIX + tile * L::TB + (e0 / 64) * (BM * 128) +
                                         t * 128;
                    uint32_t pk[16];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int unit = (e0 % 64) / 8 + u;
                        const uint4 x =
                            *reinterpret_cast<const uint4*>(row + ((unit ^ (t & 7)) << 4));
                        pk[4 * u] = x.x;
                        pk[4 * u + 1] = x.y;
                        pk[4 * u + 2] = x.z;
                        pk[4 * u + 3] = x.w;
                    }
                    tmem_st16(tA2 + (uint32_t)gc, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::BAR_QT));
            }
        }
        for (int s = 0; s < n_steps && ok; ++s) {
            // per-column values of the step's query tile (dk/dv): lane l of this warp's chunk
            // cc holds query column cb + 32 cc + l, handed to the other lanes by shuffles
            // (every lane reading all of them with broadcast loads measured slower at d = 128)
            float lse2_c[BWD_NCH], delta_c[BWD_NCH];
            const int ct = step_tile(s);
            // d = 64: this warp's lse2 then delta values, broadcast from shared memory
            float* lsw = reinterpret_cast<float*>(smem + L::OFF_LSE) + warp * (2 * BWD_CW);
            if (DKDV) {
                const int qm = step_qmat(s);
                bwd_mu(p, qm % p.Hq, mu_l2, mu_sign);
                const size_t base = (size_t)qm * p.N;
#pragma unroll
                for (int cc = 0; cc < BWD_NCH; ++cc) {
                    const int qc = ct * BM + cb + cc * 32 + (int)lane;
                    lse2_c[cc] = (qc < p.N) ? __ldg(p.lse + base + qc) * LOG2E_F - mu_l2 : 0.f;
                    delta_c[cc] = (qc < p.N) ? __ldg(p.delta + base + qc) : 0.f;
                    if (L::LSE_SMEM) {
                        lsw[cc * 32 + lane] = lse2_c[cc];
                        lsw[BWD_CW + cc * 32 + lane] = delta_c[cc];
                    }
                }
                if (L::LSE_SMEM) __syncwarp();
            }
            // allowed pairs: key j and query i with i - W < j <= i, both < N; compact key r
            // (position r * stride) and query i with r < ncomp(i), i.e. i >= r * stride + W
            //   dk/dv: this thread's key j = my, column = query ct*128 + col
            //   compact dk/dv: this thread's compact key r = my, column = query ct*128 + col
            //   dq:    this thread's query i = my, column = key ct*128 + col, or compact key
            //          c*128 + col of compact tile c = -1 - ct
            int a, bnd;  // allowed columns [a, bnd]
            if (KIND == 0) {
                const int q0 = ct * BM;
                a = my - q0;                                   // i >= j
                bnd = min(my + p.W - 1, p.N - 1) - q0;         // i <= j + W - 1, i < N
            } else if (COMPACT) {
                const int q0 = ct * BM;
                const long long first = (long long)my * p.stride + p.W;  // first reader
                a = (int)min(first - q0, (long long)BM);
                bnd = (my < p.ncomp) ? p.N - 1 - q0 : -1;
            } else if (ct < 0) {
                a = 0;
                bnd = bwd_ncomp(p, my) - 1 - (-1 - ct) * BN;
            } else {
                const int k0 = ct * BN;
                a = max(0, my - p.W + 1) - k0;
                bnd = my - k0;
            }
            if (!valid) bnd = -1;
            const uint32_t tS = tL;
            ok = wait(bar(L::BAR_SREADY), (uint32_t)s & 1u);
            if (!ok) break;
            tc_fence_after();
            // the weights of this warp's columns; a 32-column chunk wholly inside every lane's
            // allowed range (most chunks, for a window much wider than a tile) skips the mask
            float pv[BWD_CW];
#pragma unroll
            for (int cc = 0; cc < BWD_NCH; ++cc) {
                uint32_t sr[32];
                tmem_ld32(tS + (uint32_t)(cb + cc * 32), sr);
                if (!DKDV && cc == BWD_NCH - 1) {
                    // dq: S has been read; the issuer may overwrite it with S(s+1)
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(L::BAR_SFREE));
                }
                const int c0 = cb + cc * 32;
                const bool full = __all_sync(0xffffffffu, a <= c0 && bnd >= c0 + 31);
                // in two 16-column pieces, so that a piece's lse values need few registers
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float l2v[16];  // the column's lse2 (dk/dv) or the row's (dq)
                    if (!DKDV) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) l2v[u] = lse2_row;
                    } else if (L::LSE_SMEM) {
                        const float4* l4 = reinterpret_cast<const float4*>(lsw + cc * 32 + 16 * h);
#pragma unroll
                        for (int u4 = 0; u4 < 4; ++u4) {
                            const float4 x = l4[u4];
                            l2v[4 * u4] = x.x;
                            l2v[4 * u4 + 1] = x.y;
                            l2v[4 * u4 + 2] = x.z;
                            l2v[4 * u4 + 3] = x.w;
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < 16; ++u)
                            l2v[u] = __shfl_sync(0xffffffffu, lse2_c[cc], 16 * h + u);
                    }
                    if (full) {
#pragma unroll
                        for (int u = 0; u < 16; ++u)
                            pv[cc * 32 + 16 * h + u] =
                                fast_exp2(fmaf(__uint_as_float(sr[16 * h + u]), sl2, -l2v[u]));
                    } else {
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const int col = c0 + 16 * h + u;
                            const bool in = (col >= a) && (col <= bnd);
                            pv[cc * 32 + 16 * h + u] =
                                in ? fast_exp2(fmaf(__uint_as_float(sr[16 * h + u]), sl2, -l2v[u]))
                                   : 0.f;
                        }
                    }
                }
            }
            if (DKDV) {
                // P^T, packed over the first half of this warp's columns (already read)
                uint32_t pk[16];
#pragma unroll
                for (int cc = 0; cc < BWD_NCH; ++cc) {
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        pk[u] = pack_bf16x2(pv[cc * 32 + 2 * u], pv[cc * 32 + 2 * u + 1]);
                    if (mu_sign) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) pk[u] ^= mu_sign;
                    }
                    tmem_st16(tS + (uint32_t)(cb + cc * 16), pk);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::BAR_P));
            }
            // dS = P (dP - delta)
            ok = wait(bar(L::BAR_DPREADY), (uint32_t)s & 1u);
            if (!ok) break;
            tc_fence_after();
            uint32_t dsw[BWD_CW / 2];
#pragma unroll
            for (int cc = 0; cc < BWD_NCH; ++cc) {
                uint32_t dr[32];
                tmem_ld32(tDP + (uint32_t)(cb + cc * 32), dr);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float dlv[16];  // the column's delta (dk/dv) or the row's (dq)
                    if (!DKDV) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) dlv[u] = delta_row;
                    } else if (L::LSE_SMEM) {
                        const float4* d4 =
                            reinterpret_cast<const float4*>(lsw + BWD_CW + cc * 32 + 16 * h);
#pragma unroll
                        for (int u4 = 0; u4 < 4; ++u4) {
                            const float4 x = d4[u4];
                            dlv[4 * u4] = x.x;
                            dlv[4 * u4 + 1] = x.y;
                            dlv[4 * u4 + 2] = x.z;
                            dlv[4 * u4 + 3] = x.w;
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < 16; ++u)
                            dlv[u] = __shfl_sync(0xffffffffu, delta_c[cc], 16 * h + u);
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int e = cc * 32 + 16 * h + 2 * u;
                        const float d0 = pv[e] * (__uint_as_float(dr[16 * h + 2 * u]) - dlv[2 * u]);
                        const float d1 =
                            pv[e + 1] * (__uint_as_float(dr[16 * h + 2 * u + 1]) - dlv[2 * u + 1]);
                        dsw[cc * 16 + 8 * h + u] = pack_bf16x2(d0, d1);
                    }
                }
            }
            if (mu_sign) {
#pragma unroll
                for (int u = 0; u < BWD_CW / 2; ++u) dsw[u] ^= mu_sign;
            }
            // dS^T (dk/dv) or dS (dq) packed over this warp's columns of dP (already read); the
            // issuer issues dP(s+1) after the dK / dQ product that reads it
#pragma unroll
            for (int cc = 0; cc < BWD_NCH; ++cc) {
                uint32_t pk[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) pk[u] = dsw[cc * 16 + u];
                tmem_st16(tDP + (uint32_t)(cb + cc * 16), pk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::BAR_DS));
        }
        if (ok) ok = wait(bar(L::BAR_FIN), 0u);
        if (ok) {
            tc_fence_after();
            constexpr int NC = D * BWD_CW / 128;  // accumulator columns this warp stores
            const int c0 = part * NC;
            const size_t dvoff = (size_t)p.cchunks * p.B * p.Hkv * p.ncomp_pad * D;  // dk -> dv
            if (COMPACT) {
                // fp32 partial sums of this chunk (dK unscaled, as the window kernel's)
                float* pk = p.cpart + (((size_t)chunk * p.B * p.Hkv + bz) * p.ncomp_pad + my) * D;
                bwd_store_cols_f32<NC>(tA1, pk + dvoff, n_steps > 0, true, c0);
                bwd_store_cols_f32<NC>(tA2, pk, n_steps > 0, true, c0);
            } else if (DKDV) {
                const size_t row = (size_t)bz * p.N + (size_t)(valid ? my : 0);
                // a key that is also a compact key takes the compact pass's partial sums
                const float* xk = nullptr;
                if (p.cap > 0 && valid && my % p.stride == 0 && my / p.stride < p.ncomp)
                    xk = p.cpart + ((size_t)bz * p.ncomp_pad + my / p.stride) * D;
                const size_t cstride = (size_t)p.B * p.Hkv * p.ncomp_pad * D;
                if (p.dv32_out) {  // the first differential map: dV stays fp32 for the second
                    bwd_store_cols_f32<NC>(tA1, p.dv32_out + row * D, true, valid, c0);
                } else if (p.dv32_in) {  // the second map: dV of both maps, rounded once
                    bwd_store_cols<NC>(tA1, 1.f, p.dv + row * D, valid, c0,
                                          p.dv32_in + row * D, 1, 0);
                } else {  // the compact partials were summed into their first chunk
                    bwd_store_cols<NC>(tA1, 1.f, p.dv + row * D, valid, c0,
                                          xk ? xk + dvoff : nullptr, 1, cstride);
                }
                bwd_store_cols<NC>(tA2, p.scale, p.dk + row * D, valid, c0, xk, 1, cstride);
            } else {
                const size_t row = (size_t)bz * p.N + (size_t)(valid ? my : 0);
                bwd_store_cols<NC>(tA1, p.scale, p.dq + row * D, valid, c0);
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
