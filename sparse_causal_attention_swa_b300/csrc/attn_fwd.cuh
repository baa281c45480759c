// attn_fwd.cuh -- sm_103a forward kernel for causal sliding-window attention and its two
// variants (local + strided sparse, differential); a persistent grid of one CTA per SM
// walks the work items.
//
// What it computes (sources cited by page title and section):
//   * "SWA：滑动窗口注意力与跨层信息传递" §3.1: out_i = softmax_j(scale q_i.k_j + M_ij) v_j
//     with M_ij = 0 iff max(0, i-W+1) <= j <= i (0-indexed; W counts the current row),
//     each row normalised inside its own window; §4.1: work outside the window is skipped.
//   * "注意力变体——滑动窗口、稀疏、差分", "Build it" step 3: the local + strided mask adds
//     keys j = 0, s, 2s, ... <= i to the window.
//   * "Variantes de Atenção", "Atenção Diferencial": out = (A1 - lambda A2) V with two
//     softmax maps from (Q1, K1) and (Q2, K2), both causal (W = N) or both under the
//     window W (a differential head inside an SWA layer: "注意力变体", opening list, the
//     variants coexist).
//
// CTA organisation (384 threads, one CTA per SM because of TMEM and shared memory):
//   warps 0-3  softmax warpgroup of slot 0   (thread t owns query row t of the slot)
//   warps 4-7  softmax warpgroup of slot 1
//   warp 8     TMA producer (lane 0): Q tiles once, then K / V tiles into an smem ring
//   warp 9     TMEM owner; issues slot 0's MMAs: S = Q K^T and O += P V on tcgen05
//   warp 10    issues slot 1's MMAs
//   warp 11    lane 0 writes the finished output tiles out with TMA stores
// Each slot has its own issuing warp: tcgen05.mma issue blocks on a shallow queue, so a
// single issuer cannot run ahead, and its barrier bookkeeping would idle the tensor core;
// with two issuers one warp's bookkeeping overlaps the other's MMA stream.  The issuing
// warps stay converged and one elected lane performs each tcgen05 operation, which keeps
// the operands warp-uniform and makes each MMA issue about as fast as the tensor core
// executes a 128x128x16 step.  The two issuers still take turns (slot 0's batch of tile j,
// then slot 1's, then slot 0's of j+1, through the two "turn" barriers), so the tensor
// core alternates between the slots and each slot's softmax overlaps the other slot's
// MMAs; letting the issuers overlap instead drives the slots into lock step.
// setmaxnreg moves registers from the TMA / MMA warpgroup (56 per thread) to the softmax
// warpgroups (224), which hold a whole 128-key score row per thread.
// A "slot" is 128 query rows.  The two slots of a work item are either two query heads of
// one GQA group on the same rows, the two score streams of the differential variant, or
// two consecutive 128-row tiles of one head; they walk the same KV tile sequence in lock
// step so that every K / V tile is loaded once for both.
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [  0,128) S of slot 0   (P of slot 0, bf16 packed in pairs, overwrites columns [0,64))
//   [128,256) S of slot 1   (P of slot 1 in [128,192))
//   [256,256+D) O of slot 0,  [384,384+D) O of slot 1
//
// Per KV tile, slot s's MMA thread issues, in order, PV_s(j) then S_s(j+1); tcgen05 MMAs of
// one thread execute in issue order, so S_s(j+1) cannot overwrite P_s(j) before PV_s(j) has
// read it, and the commit after S_s(j+1) also covers PV_s(j).
//
// Online softmax in base 2: x = s * scale * log2(e).  The running row maximum m is only
// moved (and O, l rescaled) when the new tile's maximum exceeds it by more than 8 in the
// log2 domain; otherwise exponents stay <= 8 and p <= 256, exact in bf16 and safe in fp32.
// The final out = O / l is exact whichever maximum was used.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace swa {

constexpr int BM = 128;  // query rows per slot
constexpr int BN = 128;  // keys per KV tile
constexpr int NUM_THREADS = 384;
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;       // TMEM owner; issues the MMAs of slot 0
constexpr int MMA_WARP_1 = 10;    // issues the MMAs of slot 1
constexpr int STORE_WARP = 11;    // lane 0 issues the epilogue's TMA stores
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units

enum Mode : int { MODE_WINDOW = 0, MODE_STRIDED = 1, MODE_DIFF = 2 };

// Tile-list entry encoding (strided mode): kind in bits 24.., tile index below.
constexpr int TILE_KIND_SHIFT = 24;
constexpr int TILE_KIND_WINDOW = 0;
constexpr int TILE_KIND_STRIDED = 1;

struct KParams {
    CUtensorMap tm_q;   // queries (slot 0; both slots unless diff), view [B*Hq][N][d]
    CUtensorMap tm_k;   // keys (slot 0 / both), view [B*Hkv][N][d]
    CUtensorMap tm_v;   // values
    CUtensorMap tm_q2;  // diff: Q2
    CUtensorMap tm_k2;  // diff: K2 ; strided: compact keys, rows 0, s, 2s, ...
    CUtensorMap tm_v2;  // strided: compact values
    CUtensorMap tm_out; // output, view [B*Hq][N][d] (TMA stores of the epilogue)
    __nv_bfloat16* out;
    const int* tiles;   // strided: [n_blocks + 1] offsets, then encoded entries
    int* status;        // device status word (SWA_ERR_TIMEOUT on a watchdog abort)
    unsigned long long wait_limit_ns;
    int B, Hq, Hkv, N, W, stride;
    int n_qtiles;       // ceil(N / BM)
    int pair_mode;      // 1: both slots on the same rows; 0: consecutive row tiles of a head
    float scale_log2;   // scale * log2(e)
    float lambda;       // diff only
    const float* lambda_heads;  // diff: one lambda per query head (device), or null
    float* lse;         // window / strided: per-row log-sum-exp [B, Hq, N] (device), or null
    float scale;        // scale (natural units), for the log-sum-exp
    int strided_cap;    // strided mode: at most this many compact keys (the global-prefix
                        // form: stride 1, cap n_g); INT_MAX otherwise
    int q_off;          // window mode: query row r sits at key position r + q_off (a chunk
                        // after q_off earlier positions); 0 otherwise
    int n_items;        // work items; the grid is persistent and walks them
};

template <int D, int MODE>
struct SmemLayout {
    static constexpr int QBYTES = BM * D * 2;
    static constexpr int EBYTES = BN * D * 2;  // one ring entry: a K or V tile
    static constexpr int STAGES = (D == 128) ? 4 : 11;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_RING = 2 * QBYTES;
    // epilogue staging: one output tile, 128 rows x D bf16 as D/64 boxes of 64 columns
    // (16 KiB each, 128B-swizzled), used by one (item, slot) after another
    static constexpr int OFF_STAGE = OFF_RING + STAGES * EBYTES;
    static constexpr int STAGE_BOX = BM * 64 * 2;
    static constexpr int OFF_BAR = OFF_STAGE + (D / 64) * STAGE_BOX;
    // barriers: q_full, ring_full[S], ring_empty[S], s_full[2], p_full[2], o_final[2],
    //           lsm_ready, drain
    static constexpr int BAR_Q = 0;
    static constexpr int BAR_FULL = 1;
    static constexpr int BAR_EMPTY = 1 + STAGES;
    static constexpr int BAR_S = 1 + 2 * STAGES;
    static constexpr int BAR_P = BAR_S + 2;  // four [slot][half]: half of P is in TMEM
    static constexpr int BAR_O = BAR_P + 4;
    static constexpr int BAR_L = BAR_O + 2;
    static constexpr int BAR_DRAIN = BAR_L + 1;  // two: one per MMA issuer
    static constexpr int BAR_TURN = BAR_DRAIN + 2;  // two: "slot s may issue its next batch"
    static constexpr int BAR_QFREE = BAR_TURN + 2;  // the Q tiles may be replaced
    static constexpr int BAR_BOXF = BAR_QFREE + 1;  // the staging tile is written
    static constexpr int BAR_BOXE = BAR_BOXF + 1;   // its TMA stores have read it
    static constexpr int NBARS = BAR_BOXE + 1;
    static constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM + 4;
    static constexpr int OFF_LSM = (OFF_ABORT + 4 + 15) / 16 * 16;
    static constexpr int END = OFF_LSM + BM * 4;
    static constexpr int BYTES = END + 1024;  // slack for aligning the base to 1024
    static_assert(BYTES <= 232448, "shared memory budget");
    static_assert(EBYTES % 1024 == 0 && QBYTES % 1024 == 0 && STAGE_BOX % 1024 == 0,
                  "1024-byte tile alignment");
};

struct WorkItem {
    int b, hk;
    int h[2];    // query head of each slot
    int r0[2];   // first row of each slot
    int block;   // row-block index (tile-list row)
    int R0, R1;  // union of valid rows
};

template <int MODE>
__device__ __forceinline__ WorkItem decode_item(const KParams& p, int item) {
    WorkItem w;
    const int g = p.Hq / p.Hkv;
    if (p.pair_mode) {
        // heaviest row tiles first: the last row tile has the longest (or an equal) KV range
        const int per = (MODE == MODE_DIFF) ? p.B * p.Hq : p.B * p.Hkv * (g / 2);
        const int qt = p.n_qtiles - 1 - item / per;
        const int rem = item % per;
        if (MODE == MODE_DIFF) {
            w.b = rem / p.Hq;
            w.h[0] = w.h[1] = rem % p.Hq;
            w.hk = w.h[0] / g;
        } else {
            const int pair = rem % (g / 2);  // adjacent items share K / V tiles in L2
            const int bhk = rem / (g / 2);
            w.b = bhk / p.Hkv;
            w.hk = bhk % p.Hkv;
            w.h[0] = w.hk * g + 2 * pair;
            w.h[1] = w.h[0] + 1;
        }
        w.r0[0] = w.r0[1] = qt * BM;
        w.block = qt;
    } else {
        const int nqp = (p.n_qtiles + 1) / 2;
        const int per = p.B * p.Hq;
        const int qp = nqp - 1 - item / per;
        const int bh = item % per;
        w.b = bh / p.Hq;
        w.h[0] = w.h[1] = bh % p.Hq;
        w.hk = w.h[0] / g;
        w.r0[0] = 2 * qp * BM;
        w.r0[1] = w.r0[0] + BM;
        w.block = qp;
    }
    w.R0 = w.r0[0];
    w.R1 = min(w.r0[1] + BM - 1, p.N - 1);
    return w;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int D, int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1) attn_fwd_kernel(const __grid_constant__ KParams p) {
    using L = SmemLayout<D, MODE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + L::OFF_BAR;
    auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_ABORT);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM);
    float* lsm = reinterpret_cast<float*>(smem + L::OFF_LSM);

    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();

    // ---- the items of this CTA: a static zig-zag over rounds of gridDim.x items (items are
    // ordered heaviest first, so alternating the direction of every round evens the load)
    const int G = (int)gridDim.x;
    const int n_rounds = (p.n_items + G - 1) / G;
    auto item_of = [&](int r) -> int {
        return r * G + ((r & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
    };
    // ---- tile sequence of an item
    struct TileSeq {
        int n_tiles, kv_lo, list_off;
    };
    auto tile_seq = [&](const WorkItem& wi) -> TileSeq {
        TileSeq t;
        t.kv_lo = 0;
        t.list_off = 0;
        if (MODE == MODE_STRIDED) {
            const int nblk = p.pair_mode ? p.n_qtiles : (p.n_qtiles + 1) / 2;
            t.list_off = nblk + 1 + p.tiles[wi.block];
            t.n_tiles = p.tiles[wi.block + 1] - p.tiles[wi.block];
        } else {
            t.kv_lo = max(0, wi.R0 + p.q_off - p.W + 1) / BN;
            t.n_tiles = (wi.R1 + p.q_off) / BN - t.kv_lo + 1;
        }
        return t;
    };
    auto tile_at = [&](const TileSeq& t, int jj, int& kind, int& idx) {
        if (MODE == MODE_STRIDED) {
            const int e = p.tiles[t.list_off + jj];
            kind = e >> TILE_KIND_SHIFT;
            idx = e & ((1 << TILE_KIND_SHIFT) - 1);
        } else {
            kind = TILE_KIND_WINDOW;
            idx = t.kv_lo + jj;
        }
    };

    // ---- setup: barriers, TMEM
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(bar(L::BAR_Q), 1);
        mbar_init(bar(L::BAR_QFREE), 2);  // both issuers' last S of an item
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(bar(L::BAR_FULL + s), 1);
            mbar_init(bar(L::BAR_EMPTY + s), 2);  // released by both MMA issuers
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(L::BAR_S + s), 1);
            mbar_init(bar(L::BAR_P + 2 * s), 4);  // one arrival per softmax warp
            mbar_init(bar(L::BAR_P + 2 * s + 1), 4);
            mbar_init(bar(L::BAR_O + s), 1);
        }
        mbar_init(bar(L::BAR_BOXF), 128);
        mbar_init(bar(L::BAR_BOXE), 1);
        mbar_init(bar(L::BAR_L), 128);
        mbar_init(bar(L::BAR_DRAIN), 1);
        mbar_init(bar(L::BAR_DRAIN + 1), 1);
        mbar_init(bar(L::BAR_TURN), 1);
        mbar_init(bar(L::BAR_TURN + 1), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == PRODUCER_WARP && lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        tma_prefetch_desc(&p.tm_out);
        if (MODE != MODE_WINDOW) tma_prefetch_desc(&p.tm_k2);
        if (MODE == MODE_DIFF) tma_prefetch_desc(&p.tm_q2);
        if (MODE == MODE_STRIDED) tma_prefetch_desc(&p.tm_v2);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t lim = p.wait_limit_ns;

    // Registers: the softmax warpgroups hold a 128-key score row per thread; the TMA / MMA
    // warpgroup needs few.  Launch budget 384 x 168 = 256 x 224 + 128 x 56.
    if (warp == PRODUCER_WARP) {
        // ===================================== TMA producer
        setmaxnreg_dec<56>();
        if (lane == 0) {
            constexpr int NCH = D / 64;  // 64-column (128-byte) chunks per row
            uint32_t used_mask = 0, par_mask = 0;  // per stage: filled at least once / parity
            uint32_t st = 0, ph = 0;
            bool ok = true;
            int it = 0;  // items loaded so far
            for (int r = 0; r < n_rounds && ok; ++r) {
                const int item = item_of(r);
                if (item >= p.n_items) continue;
                const WorkItem wi = decode_item<MODE>(p, item);
                const TileSeq ts = tile_seq(wi);
                const int kmat = wi.b * p.Hkv + wi.hk;
                auto push = [&](const CUtensorMap* m, int row) -> bool {
                    if (!mbar_wait_bounded(bar(L::BAR_EMPTY + st), ph ^ 1u, abort_flag, lim))
                        return false;
                    mbar_arrive_expect_tx(bar(L::BAR_FULL + st), L::EBYTES);
                    const uint32_t dst = sbase + L::OFF_RING + st * L::EBYTES;
                    for (int c = 0; c < NCH; ++c)
                        tma_load_3d(dst + c * (BN * 128), m, bar(L::BAR_FULL + st), c * 64, row,
                                    kmat);
                    used_mask |= 1u << st;
                    par_mask = (par_mask & ~(1u << st)) | (ph << st);
                    if (++st == (uint32_t)L::STAGES) {
                        st = 0;
                        ph ^= 1u;
                    }
                    return true;
                };
                // Q tiles of both slots, once the previous item's S products have read them
                auto load_q = [&]() -> bool {
                    if (it > 0 && !mbar_wait_bounded(bar(L::BAR_QFREE), (uint32_t)(it - 1) & 1u,
                                                     abort_flag, lim))
                        return false;
                    mbar_arrive_expect_tx(bar(L::BAR_Q), 2 * L::QBYTES);
                    for (int s = 0; s < 2; ++s) {
                        const CUtensorMap* mq =
                            (MODE == MODE_DIFF && s == 1) ? &p.tm_q2 : &p.tm_q;
                        const int mat = wi.b * p.Hq + wi.h[s];
                        for (int c = 0; c < NCH; ++c)
                            tma_load_3d(sbase + L::OFF_Q + s * L::QBYTES + c * (BM * 128), mq,
                                        bar(L::BAR_Q), c * 64, wi.r0[s], mat);
                    }
                    ++it;
                    return true;
                };
                // order: K of the first tile (it can land while the previous item finishes),
                // then Q, then the rest of the item's tiles
                for (int jj = 0; jj < ts.n_tiles && ok; ++jj) {
                    int kind, idx;
                    tile_at(ts, jj, kind, idx);
                    const bool compact = (MODE == MODE_STRIDED && kind == TILE_KIND_STRIDED);
                    const CUtensorMap* mk = compact ? &p.tm_k2 : &p.tm_k;
                    const CUtensorMap* mv = compact ? &p.tm_v2 : &p.tm_v;
                    const int row = idx * BN;
                    ok = push(mk, row);
                    if (ok && MODE == MODE_DIFF) ok = push(&p.tm_k2, row);
                    if (ok && jj == 0) ok = load_q();
                    if (ok) ok = push(mv, row);
                }
            }
            // drain: every issued copy must have landed before the CTA may exit
            {
                volatile int never = 0;
                if (it > 0)
                    (void)mbar_wait_bounded(bar(L::BAR_Q), (uint32_t)(it - 1) & 1u, &never, lim);
                for (int s = 0; s < L::STAGES; ++s)
                    if (used_mask & (1u << s))
                        (void)mbar_wait_bounded(bar(L::BAR_FULL + s), (par_mask >> s) & 1u, &never,
                                                lim);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP || warp == MMA_WARP_1) {
        // ===================================== MMA issuers (one converged warp per slot)
        setmaxnreg_dec<56>();
        // All 32 lanes run the loop and wait on the barriers; each tcgen05 operation is
        // performed by one elected lane (the *_elect forms).
        const int s = (warp == MMA_WARP) ? 0 : 1;
        constexpr uint32_t ID_S = idesc_bf16_f32(BM, BN, 0);
        constexpr uint32_t ID_O = idesc_bf16_f32(BM, D, 1);
        const uint32_t ring0 = sbase + L::OFF_RING;
        // Descriptors are built once; the 14-bit start-address field holds address >> 4
        // in the low bits, so moving to another K step, chunk or ring entry is an add of
        // (byte offset >> 4) that cannot carry (shared memory addresses are < 2^18).
        const uint64_t aq = smem_desc_sw128(sbase + L::OFF_Q + s * L::QBYTES, 16, 1024);
        const uint64_t dk0 = smem_desc_sw128(ring0, 16, 1024);
        const uint64_t dv0 = smem_desc_sw128(ring0, BN * 128, 1024);
        const uint32_t tS = tmem_base + 128u * (uint32_t)s;
        const uint32_t tO = tmem_base + 256u + 128u * (uint32_t)s;
        auto issue_S = [&](int entry) {
            const uint64_t bk = dk0 + (uint64_t)(entry * (L::EBYTES >> 4));
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t offq = ((k >> 2) * (BM * 128) + (k & 3) * 32) >> 4;
                const uint32_t offk = ((k >> 2) * (BN * 128) + (k & 3) * 32) >> 4;
                mma_ss_elect(tS, aq + offq, bk + offk, ID_S, k > 0 ? 1u : 0u);
            }
        };
        // O += P V over one half of the tile's keys (k-steps 4 half .. 4 half + 3)
        auto issue_PV = [&](int entry, int half, bool acc) {
            const uint64_t bv = dv0 + (uint64_t)(entry * (L::EBYTES >> 4));
#pragma unroll
            for (int kk = 0; kk < BN / 32; ++kk) {
                const int k = half * (BN / 32) + kk;
                mma_ts_elect(tO, tS + (uint32_t)(k * 8), bv + (uint64_t)((k * 2048) >> 4), ID_O,
                             (acc || k > 0) ? 1u : 0u);
            }
        };
        // a bounded wait whose outcome every lane agrees on
        auto wait = [&](uint32_t b, uint32_t parity) -> bool {
            const bool r = mbar_wait_bounded(b, parity, abort_flag, lim);
            return __all_sync(0xffffffffu, r);
        };
        uint32_t st = 0, ph = 0;
        bool ok = true;
        auto pop = [&](int& e) -> bool {
            if (!wait(bar(L::BAR_FULL + st), ph)) return false;
            e = (int)st;
            if (++st == (uint32_t)L::STAGES) {
                st = 0;
                ph ^= 1u;
            }
            return true;
        };
        // Turn order: the slots' batches alternate, slot 0 first, across all items.  Batch
        // b of slot 0 (b >= 1) waits for the completion of phase b-1 of t[0], which slot 1
        // completes with its batch b-1; batch b of slot 1 waits for phase b of t[1], which
        // slot 0 completes with its batch b.  Neither slot can run two batches ahead, so a
        // parity wait never aliases.
        uint32_t nb = 0;  // batches this slot has issued
        auto my_turn = [&]() -> bool {
            if (s == 0) return nb == 0 ? true : wait(bar(L::BAR_TURN), (nb - 1) & 1u);
            return wait(bar(L::BAR_TURN + 1), nb & 1u);
        };
        uint32_t np = 0;  // P phases consumed
        // Both issuers pop every ring entry (in the producer's order) and release every
        // entry they popped, so each empty barrier gets its two arrivals; an entry this
        // slot does not read (the other stream's K in the differential call) is released
        // after this warp's earlier MMAs, which is merely conservative.
        int it = 0;
        for (int r = 0; r < n_rounds && ok; ++r) {
            const int item = item_of(r);
            if (item >= p.n_items) continue;
            const TileSeq ts = tile_seq(decode_item<MODE>(p, item));
            int kA = 0, kB = 0;
            ok = wait(bar(L::BAR_Q), (uint32_t)it & 1u);
            if (ok) ok = pop(kA);
            if (ok && MODE == MODE_DIFF) ok = pop(kB);
            if (ok) ok = my_turn();
            if (!ok) break;
            tc_fence_after();
            issue_S((MODE == MODE_DIFF && s == 1) ? kB : kA);
            mma_commit_elect(bar(L::BAR_S + s));
            if (ts.n_tiles == 1) mma_commit_elect(bar(L::BAR_QFREE));
            mma_commit_elect(bar(L::BAR_EMPTY + kA));
            if (MODE == MODE_DIFF) mma_commit_elect(bar(L::BAR_EMPTY + kB));
            mbar_arrive_elect(bar(L::BAR_TURN + (s ^ 1)));
            ++nb;
            for (int jj = 0; jj < ts.n_tiles && ok; ++jj) {
                int ve = 0, nA = 0, nB = 0;
                const bool more = jj + 1 < ts.n_tiles;
                ok = pop(ve);
                if (ok && more) {
                    ok = pop(nA);
                    if (ok && MODE == MODE_DIFF) ok = pop(nB);
                }
                // Both the slot's P and its turn are needed; wait first on the one that
                // usually completes first (slot 0: its turn, slot 1: its P), so the second
                // wait's latency is the only one left on the critical path.  P arrives in two
                // halves; the first half's products start while the softmax finishes the
                // second.
                if (s == 0) {
                    if (ok) ok = my_turn();
                    if (ok) ok = wait(bar(L::BAR_P + 2 * s), np & 1u);
                } else {
                    if (ok) ok = wait(bar(L::BAR_P + 2 * s), np & 1u);
                    if (ok) ok = my_turn();
                }
                if (!ok) break;
                tc_fence_after();
                issue_PV(ve, 0, jj > 0);
                ok = wait(bar(L::BAR_P + 2 * s + 1), np & 1u);
                ++np;
                if (!ok) break;
                tc_fence_after();
                issue_PV(ve, 1, true);
                if (more) {
                    issue_S((MODE == MODE_DIFF && s == 1) ? nB : nA);
                    mma_commit_elect(bar(L::BAR_S + s));
                    // the item's last S product: its Q tile may be replaced once it is done
                    if (jj + 2 == ts.n_tiles) mma_commit_elect(bar(L::BAR_QFREE));
                } else {
                    mma_commit_elect(bar(L::BAR_O + s));
                }
                mbar_arrive_elect(bar(L::BAR_TURN + (s ^ 1)));
                ++nb;
                mma_commit_elect(bar(L::BAR_EMPTY + ve));
                if (more) {
                    mma_commit_elect(bar(L::BAR_EMPTY + nA));
                    if (MODE == MODE_DIFF) mma_commit_elect(bar(L::BAR_EMPTY + nB));
                }
            }
            ++it;
        }
        // drain: all MMAs this warp issued must complete before TMEM is released
        __syncwarp();
        mma_commit_elect(bar(L::BAR_DRAIN + s));
        volatile int never = 0;
        (void)mbar_wait_bounded(bar(L::BAR_DRAIN + s), 0, &never, lim);
        __syncwarp();
    } else if (warp < 8) {
        // ===================================== softmax warpgroups
        setmaxnreg_inc<224>();
        const int s = (int)(warp >> 2);
        const int wq = (int)(warp & 3);
        const int trow = wq * 32 + (int)lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem_base + lane_off + (uint32_t)(s * 128);
        const uint32_t tO = tmem_base + lane_off + 256u + (uint32_t)(s * 128);
        const float sl2 = p.scale_log2;
        bool ok = true;
        uint32_t ns = 0;  // S phases consumed
        int it = 0;
        for (int r = 0; r < n_rounds && ok; ++r) {
            const int item = item_of(r);
            if (item >= p.n_items) continue;
            const WorkItem wi = decode_item<MODE>(p, item);
            const TileSeq ts = tile_seq(wi);
            const int row = wi.r0[s] + trow;
            const int rowk = row + p.q_off;  // the query's key position
            const int lo_i = max(0, rowk - p.W + 1);
            // compact keys of this row: the multiples of the stride before its window start
            // (at most strided_cap of them: the global prefix j < n_g when the stride is 1)
            const int lo_strided =
                (MODE == MODE_STRIDED) ? min((lo_i + p.stride - 1) / p.stride, p.strided_cap) : 0;
            float m = -INFINITY, l = 0.f;
            for (int jj = 0; jj < ts.n_tiles; ++jj) {
                ok = mbar_wait_bounded(bar(L::BAR_S + s), ns & 1u, abort_flag, lim);
                ++ns;
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                // the whole 128-key score row of this thread, one TMEM load
                uint32_t xr[BN];
                tmem_ld128(tS, xr);
                // allowed columns of this row in this tile: [a, bnd]
                int kind, idx;
                tile_at(ts, jj, kind, idx);
                int a, bnd;
                if (MODE == MODE_STRIDED && kind == TILE_KIND_STRIDED) {
                    a = 0;
                    bnd = lo_strided - idx * BN - 1;
                } else {
                    const int c0 = idx * BN;
                    a = lo_i - c0;
                    bnd = rowk - c0;
                }
                // Mask, on edge tiles only: columns outside [a, bnd] become -inf.  Usually only
                // one side cuts the tile (the diagonal tile: t <= bnd; the window-start tile:
                // t >= a), which needs one compare per element.
                if (a > 0 || bnd < BN - 1) {
                    if (a <= 0) {
#pragma unroll
                        for (int t = 0; t < BN; ++t)
                            xr[t] = (t <= bnd) ? xr[t] : __float_as_uint(-INFINITY);
                    } else if (bnd >= BN - 1) {
#pragma unroll
                        for (int t = 0; t < BN; ++t)
                            xr[t] = (t >= a) ? xr[t] : __float_as_uint(-INFINITY);
                    } else {
#pragma unroll
                        for (int t = 0; t < BN; ++t)
                            xr[t] = (t >= a && t <= bnd) ? xr[t] : __float_as_uint(-INFINITY);
                    }
                }
                // row maximum: eight independent 3-input max chains, then a short tree
                float mc[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float v = __uint_as_float(xr[c * 16]);
#pragma unroll
                    for (int u = 1; u < 15; u += 2)
                        v = fmax3(v, __uint_as_float(xr[c * 16 + u]),
                                  __uint_as_float(xr[c * 16 + u + 1]));
                    mc[c] = fmaxf(v, __uint_as_float(xr[c * 16 + 15]));
                }
                const float mt = fmax3(fmax3(mc[0], mc[1], mc[2]), fmax3(mc[3], mc[4], mc[5]),
                                       fmaxf(mc[6], mc[7]));
                const float m_new = fmaxf(m, mt);
                const bool need = (m_new - m) * sl2 > RESCALE_THRESHOLD;
                const bool rescale = __any_sync(0xffffffffu, need);
                float alpha = 1.f;
                if (rescale) {
                    alpha = (m_new == -INFINITY) ? 1.f : fast_exp2((m - m_new) * sl2);
                    l *= alpha;
                    m = m_new;
                }
                // O is complete up to tile jj-1 here (its PV was issued before this tile's S);
                // a rescale must reach O before the first half of P is published
                if (rescale && jj > 0) {
                    uint32_t rr[32];
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        tmem_ld32(tO + c * 32, rr);
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            rr[t] = __float_as_uint(__uint_as_float(rr[t]) * alpha);
                        tmem_st32(tO + c * 32, rr);
                    }
                }
                const float ms = (m == -INFINITY) ? 0.f : m * sl2;
                // P = exp2(x * scale * log2 e - m * scale * log2 e): the argument two lanes at
                // a time (packed fma), four packed partial row sums, bf16 pairs stored to TMEM
                // per 64-column half, each half published (one arrival per warp) as soon as
                // it is in TMEM
                const uint64_t sl2x2 = f32x2_pack(sl2, sl2);
                const uint64_t nmsx2 = f32x2_pack(-ms, -ms);
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int c = 0; c < BN / 64; ++c) {
                    uint32_t pk[32];
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const int e = c * 64 + 2 * t;
                        const uint64_t z = f32x2_fma(
                            f32x2_pack(__uint_as_float(xr[e]), __uint_as_float(xr[e + 1])), sl2x2,
                            nmsx2);
                        float z0, z1;
                        f32x2_unpack(z, z0, z1);
                        const float p0 = fast_exp2(z0);
                        const float p1 = fast_exp2(z1);
                        acc[t & 3] = f32x2_add(acc[t & 3], f32x2_pack(p0, p1));
                        pk[t] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32(tS + c * 32, pk);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(L::BAR_P + 2 * s + c));
                }
                {
                    const uint64_t s01 = f32x2_add(acc[0], acc[1]);
                    const uint64_t s23 = f32x2_add(acc[2], acc[3]);
                    float u0, u1;
                    f32x2_unpack(f32x2_add(s01, s23), u0, u1);
                    l += u0 + u1;
                }
            }
            if (!ok) break;
            // ---- epilogue of the item.  Its TMEM reads of O precede this slot's next P
            // arrival, and the next item's first O product is issued only after that.
            ok = mbar_wait_bounded(bar(L::BAR_O + s), (uint32_t)it & 1u, abort_flag, lim);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
            // log-sum-exp of the row's scores: l sums exp2((x - m) scale log2 e), so
            // ln sum_j exp(scale x_j) = m scale + ln l for whichever maximum m was used
            if (MODE != MODE_DIFF && p.lse != nullptr && row < p.N)
                p.lse[(size_t)(wi.b * p.Hq + wi.h[s]) * p.N + row] =
                    (l > 0.f) ? m * p.scale + logf(l) : -INFINITY;
            // Differential: slot 0 writes out O1 / l1 - lambda O2 / l2, reading slot 1's O2 and
            // 1 / l2 (through lsm).  The turn order keeps both intact until then: slot 1's next
            // P V product (which overwrites O2) is issued after slot 0's, and slot 0 publishes
            // the P it needs only after this epilogue; slot 1 reaches its next lsm write even
            // later.
            if (MODE == MODE_DIFF && s == 1) {
                lsm[trow] = inv_l;
                mbar_arrive(bar(L::BAR_L));
            } else {
                float inv_l2 = 0.f;
                if (MODE == MODE_DIFF) {
                    ok = mbar_wait_bounded(bar(L::BAR_L), (uint32_t)it & 1u, abort_flag, lim);
                    if (ok)
                        ok = mbar_wait_bounded(bar(L::BAR_O + 1), (uint32_t)it & 1u, abort_flag,
                                               lim);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    inv_l2 = lsm[trow] * (p.lambda_heads ? p.lambda_heads[wi.h[0]] : p.lambda);
                }
                // O / l (differential: O1 / l1 - lambda O2 / l2) to bf16 into the staging tile
                // (128-byte box rows, 16-byte unit u stored at u ^ (row & 7)); the store warp
                // writes it out with TMA, which drops the rows past N.  Uses of the staging
                // tile alternate between the slots, item after item: use u waits until the
                // stores of use u-1 have read it.
                const uint32_t tO2 = tmem_base + lane_off + 384u;
                const uint32_t use = (MODE == MODE_DIFF) ? (uint32_t)it : 2u * (uint32_t)it + (uint32_t)s;
                if (use > 0)
                    ok = mbar_wait_bounded(bar(L::BAR_BOXE), (use - 1) & 1u, abort_flag, lim);
                if (!ok) break;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(tO + c * 32, rr);
                    float y[32];
#pragma unroll
                    for (int t = 0; t < 32; ++t) y[t] = __uint_as_float(rr[t]) * inv_l;
                    if (MODE == MODE_DIFF) {
                        tmem_ld32(tO2 + c * 32, rr);
#pragma unroll
                        for (int t = 0; t < 32; ++t) y[t] -= __uint_as_float(rr[t]) * inv_l2;
                    }
                    const uint32_t brow = sbase + L::OFF_STAGE + (uint32_t)((c >> 1) * L::STAGE_BOX) +
                                          (uint32_t)trow * 128u;
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        const uint32_t u = (uint32_t)((c & 1) * 4 + v4);
                        st_shared_v4(brow + ((u ^ (uint32_t)(trow & 7)) << 4),
                                     pack_bf16x2(y[v4 * 8 + 0], y[v4 * 8 + 1]),
                                     pack_bf16x2(y[v4 * 8 + 2], y[v4 * 8 + 3]),
                                     pack_bf16x2(y[v4 * 8 + 4], y[v4 * 8 + 5]),
                                     pack_bf16x2(y[v4 * 8 + 6], y[v4 * 8 + 7]));
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(bar(L::BAR_BOXF));
            }
            if (!ok) break;
            ++it;
        }
    } else {
        // ===================================== TMA stores of the epilogue (lane 0)
        setmaxnreg_dec<56>();
        if (lane == 0) {
            bool ok = true;
            uint32_t use = 0;
            for (int r = 0; r < n_rounds && ok; ++r) {
                const int item = item_of(r);
                if (item >= p.n_items) continue;
                const WorkItem wi = decode_item<MODE>(p, item);
                constexpr int NOUT = (MODE == MODE_DIFF) ? 1 : 2;  // output tiles per item
                for (int s = 0; s < NOUT && ok; ++s, ++use) {
                    ok = mbar_wait_bounded(bar(L::BAR_BOXF), use & 1u, abort_flag, lim);
                    if (!ok) break;
                    if (wi.r0[s] < p.N) {
                        for (int c = 0; c < D / 64; ++c)
                            tma_store_3d(&p.tm_out, sbase + L::OFF_STAGE + c * L::STAGE_BOX, c * 64,
                                         wi.r0[s], wi.b * p.Hq + wi.h[s]);
                    }
                    bulk_commit_group();
                    bulk_wait_read_all();
                    mbar_arrive(bar(L::BAR_BOXE));
                }
            }
            bulk_wait_all();  // the output is written before the CTA exits
        }
        __syncwarp();
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicExch(p.status, 6 /* SWA_ERR_TIMEOUT */);
}

// One CTA waits on a barrier nobody arrives at; the bounded wait must run out and report.
__global__ void watchdog_selftest_kernel(int* status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t b;
    __shared__ int abort_word;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&b), 1);
        abort_word = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool ok = mbar_wait_bounded(smem_u32(&b), 0, &abort_word, limit_ns);
        if (!ok) atomicExch(status, 6 /* SWA_ERR_TIMEOUT */);
    }
}

}  // namespace swa
