/*
 * swa_b300.h -- C ABI of the B300 (sm_103a) sliding-window / sparse / differential
 * causal attention library (libswa_b300.so): the forward calls, decode and chunked prefill
 * against a rolling KV cache, and the backward pass of causal SWA.
 *
 * Sources, cited by page title and section:
 *   [SWA]  "SWA：滑动窗口注意力与跨层信息传递" (lizn-zn.github.io): §1 (the window W
 *          counts the current position; FlashAttention window_size = (W-1, 0)),
 *          §3.1 (window set N_W(i) = {j : max(1, i-W+1) <= j <= i}, mask M^SWA and
 *          Attention_SWA = softmax(Q K^T / sqrt(d_k) + M^SWA) V, row-wise softmax),
 *          §4.1 (skip the work outside the window).
 *   [AV]   "注意力变体——滑动窗口、稀疏、差分" (ai-engineering.com.cn), "Build it"
 *          step 2 (sliding-window causal mask), step 3 (local + strided mask),
 *          step 4 (differential attention); exercises 2-4 (training with SWA layers,
 *          a learnable lambda per head).
 *   [AVpt] "Variantes de Atenção — Janela Deslizante, Esparsa, Diferencial"
 *          (ai-engineering.academy), "Atenção Diferencial": A1 = softmax(Q1 K1^T / sqrt d),
 *          A2 = softmax(Q2 K2^T / sqrt d), DiffAttn = (A1 - lambda A2) V.
 *
 * Common conventions for the three compute calls:
 *   - Tensors are bf16, contiguous, layout [B, H, N, d]: q, q1, q2 and out have
 *     H = Hq heads; k, k1, k2 and v have H = Hkv heads.  Query head h reads
 *     key/value head h / (Hq / Hkv) (grouped-query attention).
 *   - Rows are 0-indexed: query i may read key j iff max(0, i - W + 1) <= j <= i.
 *     W >= N gives full causal attention; W = 1 lets each row read only itself.
 *   - scale multiplies q . k before the softmax (the pages use 1 / sqrt(d)).
 *   - All pointers are DEVICE pointers owned by the caller; out must not overlap an
 *     input.  Every pointer must be 16-byte aligned.  The call is asynchronous on
 *     `stream` (a cudaStream_t passed as void*; NULL = the legacy default stream) and
 *     does not synchronise.  Accumulation is fp32; out is rounded to bf16 (RNE).
 *   - d must be 64 or 128; N * d * 2 bytes per head must fit the TMA limits
 *     (N < 2^31).  The device must be sm_103 (B300).
 *   - The library keeps process-lifetime state per device (kernel attributes, a
 *     cached strided tile list); it performs no per-call allocation except the
 *     first strided call for a new (N, W, stride) shape, which builds and caches
 *     that shape's tile list.
 *   - Errors are returned as swa_status codes; nothing is thrown across the ABI.
 *     Argument errors are detected on the host before anything is launched.
 */
#ifndef SWA_B300_H
#define SWA_B300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum swa_status {
    SWA_OK = 0,
    SWA_ERR_NULL = 1,        /* a required pointer is NULL */
    SWA_ERR_SHAPE = 2,       /* B, Hq, Hkv, N < 1; W < 1; stride < 1; Hq % Hkv != 0; N too large */
    SWA_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
    SWA_ERR_UNSUPPORTED = 4, /* d not in {64, 128}, or the current device is not sm_103 */
    SWA_ERR_CUDA = 5,        /* a CUDA runtime / driver call failed (launch, attribute, map) */
    SWA_ERR_TIMEOUT = 6,     /* a kernel-side bounded wait ran out (read by swa_device_status) */
    SWA_ERR_VALUE = 7,       /* scale not finite and > 0, or lambda not finite */
    SWA_ERR_TOO_LARGE = 8    /* a fixed capacity (the no-alloc tile list, a decode or backward workspace) is too small */
} swa_status;

/* Capacity, in int entries (256 KiB), of the fixed device array that
 * strided_attn_fwd_noalloc keeps its tile list in. */
#define SWA_NOALLOC_TILE_CAPACITY 65536

/*
 * Causal sliding-window attention forward ([SWA] §3.1; [AV] step 2):
 *   out[b, h, i, :] = sum_{j = max(0, i-W+1)}^{i} softmax_j(scale * q_i . k_j) v_j
 * with each row's softmax normalised over its own window.  W >= N is full causal.
 */
int swa_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                 int Hkv, int N, int d, int W, float scale, void* stream);

/*
 * swa_attn_fwd that also writes each row's log-sum-exp, the normaliser of its softmax:
 *   lse[b, h, i] = ln sum_{j in the window of i} exp(scale * q_i . k_j)     (float32)
 * (what a backward pass or a combination of partial attention results needs).
 * lse: float32 [B, Hq, N] device, 4-byte aligned; NULL behaves as swa_attn_fwd.
 */
int swa_attn_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                     int Hq, int Hkv, int N, int d, int W, float scale, void* stream);

/*
 * Local + strided sparse causal attention forward ([AV] step 3): row i reads the
 * window keys max(0, i-W+1) <= j <= i and every key j = 0, stride, 2*stride, ... <= i
 * (absolute multiples of stride; a key in both sets counts once).
 * The first call for a new (N, W, stride) builds and caches a device tile list.
 */
int strided_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                     int Hkv, int N, int d, int W, int stride, float scale, void* stream);

/* strided_attn_fwd that also writes each row's log-sum-exp over its mask (as swa_attn_fwd_lse). */
int strided_attn_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse,
                         int B, int Hq, int Hkv, int N, int d, int W, int stride, float scale,
                         void* stream);

/*
 * Sliding window plus a global prefix ([AV] "稀疏 / 块注意力": Longformer-style global
 * tokens such as [CLS] attend to all and are attended by all): row i reads its window
 * max(0, i-W+1) <= j <= i and every key j < n_global with j <= i, a key in both counted once.
 * Under the causal mask a global row (i < n_global) reads every j <= i.  n_global >= 0
 * (0 is swa_attn_fwd; n_global >= N is full causal).  Runs the strided kernel with stride 1
 * and the compact keys capped at n_global; the first call for a new (N, W, n_global) builds
 * and caches a device tile list.
 */
int global_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                    int Hkv, int N, int d, int W, int n_global, float scale, void* stream);

/*
 * Differential causal attention forward ([AVpt] "Atenção Diferencial"; [AV] step 4):
 *   out = (softmax_causal(scale Q1 K1^T) - lambda softmax_causal(scale Q2 K2^T)) V.
 * q1, q2, out: Hq heads; k1, k2, v: Hkv heads.  Both maps are full causal.
 */
int diff_attn_fwd(const void* q1, const void* k1, const void* q2, const void* k2,
                  const void* v, float lambda, void* out, int B, int Hq, int Hkv, int N, int d,
                  float scale, void* stream);

/*
 * Differential causal attention with one lambda per query head (the attention-variants
 * lesson's exercise 4, "a learnable lambda per head"): head h of out is
 *   (softmax_causal(scale Q1_h K1^T) - lambda[h] softmax_causal(scale Q2_h K2^T)) V.
 * lambda: float32 [Hq] DEVICE array (read by the kernel, so a training loop can update it
 * in place), 4-byte aligned.  Everything else as diff_attn_fwd.
 */
int diff_attn_fwd_heads(const void* q1, const void* k1, const void* q2, const void* k2,
                        const void* v, const float* lambda, void* out, int B, int Hq, int Hkv,
                        int N, int d, float scale, void* stream);

/*
 * A differential head inside an SWA layer ([AV] opening list: the variants coexist, most
 * layers SWA with a few differential heads; [AVpt] "Atenção Diferencial" for the form):
 * both maps take the window mask of width W,
 *   out_i = sum_j (a1_ij - lambda_h a2_ij) v_j,  a_ij = softmax over max(0, i-W+1) <= j <= i.
 * W >= 1 (W >= N is diff_attn_fwd / diff_attn_fwd_heads; W < 1 returns SWA_ERR_SHAPE).
 * lambda_heads: float32 [Hq] DEVICE array, 4-byte aligned, or NULL to use the scalar lambda
 * for every head.  Layouts, ownership and errors as diff_attn_fwd.
 */
int diff_swa_attn_fwd(const void* q1, const void* k1, const void* q2, const void* k2,
                      const void* v, float lambda, const float* lambda_heads, void* out, int B,
                      int Hq, int Hkv, int N, int d, int W, float scale, void* stream);

/*
 * strided_attn_fwd without any device allocation.  The pages have no counterpart to
 * this call; it exists for callers that cannot call cudaMalloc, for example code that
 * runs under an external memory manager or an allocator that forbids foreign device
 * allocations, or a process that must not grow its device footprint after start-up.
 * Same arguments, semantics and result as strided_attn_fwd.  Instead of the cached,
 * cudaMalloc'ed tile list, the call rebuilds the list on `stream` with a small device
 * kernel inside one fixed file-scope device array of SWA_NOALLOC_TILE_CAPACITY ints
 * (256 KiB, held by every GPU that loads the library until the process exits).
 *   - The first call on a device looks up that array's device address (once per
 *     device); make that first call before any stream capture.
 *   - A problem whose tile list needs more than SWA_NOALLOC_TILE_CAPACITY entries is
 *     rejected with SWA_ERR_TOO_LARGE before anything is launched.  The list holds
 *     ceil(N / R) + 1 offsets plus, per block of R rows (R = 128 when Hq / Hkv is even,
 *     else 256), the strided tiles before the block's windows and its window tiles.
 *   - Every call shares the one array: calls whose kernels may overlap on the GPU
 *     (different streams without ordering between them) race on it and must not be
 *     issued; calls on one stream are ordered and safe.
 *   - The call itself allocates nothing: no cudaMalloc, no cudaFree, no allocating
 *     library routine.
 */
int strided_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, int B,
                             int Hq, int Hkv, int N, int d, int W, int stride, float scale,
                             void* stream);

/*
 * Decode step against a rolling W-slot KV cache ([SWA] §4.2; window of [SWA] §3.1).
 * The cache of every (sequence b, KV head) holds W rows; the key and value of absolute
 * position j live in slot j mod W (the note's 1-indexed slot (i-1) mod W), written there by
 * swa_cache_append or by the caller.  For each sequence b the query at absolute position
 * t = pos[b] reads the positions max(0, t-W+1) .. t, i.e. the slots 0 .. min(t, W-1):
 *   out[b, h, :] = sum over those slots s of softmax_s(scale * q[b, h] . k_cache[b, h/g, s])
 *                  * v_cache[b, h/g, s]          (g = Hq / Hkv)
 * The slot order is not the time order; the softmax over the window does not depend on
 * it (positional encodings must already be applied to the cached keys).
 *   q, out:             bf16 [B, Hq, d] device, contiguous
 *   k_cache, v_cache:   bf16 [B, Hkv, W, d] device, contiguous (only the window slots are
 *                       read; the others may hold anything)
 *   pos:                int32 [B] device (read by the kernels, so the call can be
 *                       captured in a CUDA graph and replayed with new positions); a
 *                       negative position gives a zero output row
 *   workspace:          device scratch of at least swa_decode_workspace_bytes(B, Hq, W, d)
 *                       bytes, 256-byte aligned, owned by the caller; calls that may run
 *                       at the same time need separate workspaces
 * Hq / Hkv must be at most 16; d 64 or 128.  Two kernels are launched on `stream`
 * (split-K over the slots, then the combine).  Errors as for the other calls;
 * SWA_ERR_TOO_LARGE if workspace_bytes is too small.
 */
size_t swa_decode_workspace_bytes(int B, int Hq, int W, int d);

/*
 * Backward pass of causal sliding-window attention (the forward of [SWA] §3.1; training
 * with SWA layers is [AV] exercises 2-3).  With dout = dL/dout and a_ij the forward's
 * softmax weights over the window max(0, i-W+1) <= j <= i:
 *   dv_j = sum_i a_ij dout_i
 *   ds_ij = a_ij (dout_i . v_j - delta_i),   delta_i = dout_i . out_i
 *   dq_i = scale sum_j ds_ij k_j,            dk_j = scale sum_i ds_ij q_i
 * dk and dv of a KV head sum over the Hq / Hkv query heads that read it.
 *   q, out, dout, dq:  bf16 [B, Hq, N, d] device, contiguous, 16-byte aligned
 *   k, v, dk, dv:      bf16 [B, Hkv, N, d] device, contiguous, 16-byte aligned
 *   lse:               fp32 [B, Hq, N] device, the row log-sum-exp that swa_attn_fwd_lse
 *                      wrote with the same q, k, W and scale (a_ij = exp(scale q_i.k_j - lse_i))
 *   out:               the forward output of that call
 *   workspace:         device scratch of at least swa_attn_bwd_workspace_bytes(B, Hq, N)
 *                      bytes, 16-byte aligned, owned by the caller (it receives delta)
 * dq, dk and dv are overwritten (not accumulated into).  Three kernels run on `stream`: delta,
 * then dk / dv (one CTA per 128-key tile), then dq (one CTA per 128-row tile); the result is
 * deterministic.  W >= 1 (W > N is N); B * Hq <= 65535; d 64 or 128.  Errors as for
 * swa_attn_fwd; SWA_ERR_TOO_LARGE if workspace_bytes is too small.
 */
size_t swa_attn_bwd_workspace_bytes(int B, int Hq, int N);
int swa_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                 int d, int W, float scale, void* workspace, size_t workspace_bytes,
                 void* stream);
/*
 * Backward pass of local + strided sparse causal attention ([AV] step 3; the same chain rule
 * as swa_attn_bwd): row i reads its window max(0, i-W+1) <= j <= i and the keys
 * j = 0, stride, 2*stride, ... before the window; a_ij is the forward's weight over that set
 * (lse from strided_attn_fwd_lse with the same q, k, W, stride and scale).  Arguments, layouts,
 * ownership and errors as swa_attn_bwd, with
 *   workspace: at least strided_attn_bwd_workspace_bytes(B, Hq, Hkv, N, d, W, stride) bytes;
 *              it receives delta and fp32 partial sums of the keys j = 0, stride, ... .
 * Four kernels run on `stream`: delta, the dk / dv of the strided keys (their readers are every
 * row past their window, walked in chunks), the window dk / dv (which adds those partial sums
 * before rounding), then dq (each row tile's strided keys, then its window).  Deterministic.
 */
size_t strided_attn_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int W,
                                        int stride);
int strided_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                     int Hq, int Hkv, int N, int d, int W, int stride, float scale,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * global_attn_fwd that also writes each row's log-sum-exp over its mask (as swa_attn_fwd_lse).
 */
int global_attn_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse,
                        int B, int Hq, int Hkv, int N, int d, int W, int n_global, float scale,
                        void* stream);

/*
 * Backward pass of the window plus a global prefix ([AV] "稀疏 / 块注意力", the mask of
 * global_attn_fwd): row i reads its window and every key j < n_global with j <= i.  lse from
 * global_attn_fwd_lse with the same arguments.  As strided_attn_bwd with the prefix in place
 * of the strided keys; workspace: at least global_attn_bwd_workspace_bytes(B, Hq, Hkv, N, d, W,
 * n_global) bytes.  n_global >= 0 (0 is swa_attn_bwd; n_global >= N is full causal).
 */
size_t global_attn_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int W,
                                       int n_global);
int global_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                    const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                    int Hq, int Hkv, int N, int d, int W, int n_global, float scale,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass of differential attention ([AVpt] "Atenção Diferencial", out = (A1 - lambda_h
 * A2) V; both maps under the window W as in diff_swa_attn_fwd, W >= N causal as in
 * diff_attn_fwd / diff_attn_fwd_heads).  With dout = dL/dout and da_ij = dout_i . v_j:
 *   dv_j  = sum_i (a1_ij - lambda_h a2_ij) dout_i
 *   dq1_i = scale sum_j a1_ij (da_ij - dout_i . out1_i) k1_j,   dk1 likewise
 *   dq2_i = -lambda_h scale sum_j a2_ij (da_ij - dout_i . out2_i) k2_j,   dk2 likewise
 *   dlambda_h = -sum over batches and rows of dout_i . out2_i
 * where out1 = A1 V and out2 = A2 V with their row log-sum-exps lse1, lse2 are what
 * swa_attn_fwd_lse(q1, k1, v, ...) and swa_attn_fwd_lse(q2, k2, v, ...) write with the same
 * W and scale (the training forward runs those two calls; diff_swa_attn_fwd gives out itself).
 *   lambda / lambda_heads: as diff_swa_attn_fwd (lambda_heads: float32 [Hq] device, or NULL)
 *   dlambda:   float32 [Hq] device (4-byte aligned), each head's lambda gradient, or NULL
 *   q1, q2, out1, out2, dout, dq1, dq2: bf16 [B, Hq, N, d];  k1, k2, v, dk1, dk2, dv: bf16
 *   [B, Hkv, N, d] (dk and dv of a KV head sum over its query heads);  lse1, lse2: fp32 [B, Hq, N]
 *   workspace: at least diff_attn_bwd_workspace_bytes(B, Hq, Hkv, N, d) bytes, 16-byte aligned
 *              (two deltas and map 1's fp32 dv)
 * Map 2 runs the SWA backward kernels with each step's weights scaled by -lambda_h; dv of the
 * two maps is summed in fp32 and rounded once.  Deterministic.  Errors as swa_attn_bwd.
 */
size_t diff_attn_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d);
int diff_attn_bwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                  float lambda, const float* lambda_heads, const void* out1, const float* lse1,
                  const void* out2, const float* lse2, const void* dout, void* dq1, void* dk1,
                  void* dq2, void* dk2, void* dv, float* dlambda, int B, int Hq, int Hkv, int N,
                  int d, int W, float scale, void* workspace, size_t workspace_bytes,
                  void* stream);

int swa_decode_fwd(const void* q, const void* k_cache, const void* v_cache, const int* pos,
                   void* out, int B, int Hq, int Hkv, int W, int d, float scale, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * Rolling-cache update ([SWA] §4.2): writes n new rows per (sequence b, KV head h),
 * k_new[b, h, r, :] and v_new[b, h, r, :] (bf16 [B, Hkv, n, d] device), which hold positions
 * pos[b] + r, into slot (pos[b] + r) mod W of k_cache / v_cache (bf16 [B, Hkv, W, d] device),
 * overwriting the positions that left the window.  Of a block longer than W only the last W
 * rows are written.  pos: int32 [B] device; a negative position writes nothing.  n = 1 is
 * the per-token update of a decode step.  One kernel on `stream`.
 */
int swa_cache_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                     const int* pos, int B, int Hkv, int W, int d, int n, void* stream);

/*
 * Chunked prefill ([SWA] §4.3: the queries of a chunk need different windows, across the
 * history and the chunk, under the local causal mask).  The queries q (bf16 [B, Hq, C, d])
 * are the LAST C positions of a contiguous key/value context k, v (bf16 [B, Hkv, L, d],
 * C <= L): query row c sits at key position L - C + c and reads the keys
 * max(0, L-C+c-W+1) .. L-C+c.  out: bf16 [B, Hq, C, d].  With C = L this is swa_attn_fwd.
 * For a rolling cache, build the context with swa_cache_gather (the W-1 positions before the
 * chunk, in time order) followed by the chunk's own keys and values, then append the chunk
 * with swa_cache_append (n = C).  Same kernel, layout and error rules as swa_attn_fwd.
 */
int swa_chunk_fwd(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                  int Hkv, int C, int L, int d, int W, float scale, void* stream);

/*
 * Copy positions pos0 - nctx .. pos0 - 1 (0 <= nctx <= min(W, pos0)) out of the rolling caches
 * (slot = position mod W, [SWA] §4.2), in time order, into rows 0 .. nctx-1 of the contiguous
 * context buffers k_ctx, v_ctx (bf16 [B, Hkv, ctx_rows, d] device, ctx_rows >= nctx).
 * pos0 is the same for every sequence of the batch.  One kernel on `stream`.
 */
int swa_cache_gather(const void* k_cache, const void* v_cache, void* k_ctx, void* v_ctx, int B,
                     int Hkv, int W, int d, int pos0, int nctx, int ctx_rows, void* stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char* swa_status_string(int status);

/*
 * The cause of the calling thread's last SWA_ERR_CUDA: the CUDA call that failed and its
 * error name (thread-local storage, valid until the thread's next failing call; "" if none).
 */
const char* swa_last_error_detail(void);

/*
 * Synchronise `stream`, then read and clear the library's device status word on the
 * current device.  Returns SWA_OK, SWA_ERR_TIMEOUT if a kernel's bounded wait ran out
 * since the last call (that kernel wrote no output rows it could not finish), or
 * SWA_ERR_CUDA if the synchronisation itself failed.
 */
int swa_device_status(void* stream);

/*
 * Self-test of the kernel watchdog: launches one CTA that waits on a barrier nobody
 * arrives at, with a wait limit of `limit_us` microseconds (1..1000000).  The wait runs
 * out, the kernel records SWA_ERR_TIMEOUT in the device status word and returns.
 * Asynchronous; read the outcome with swa_device_status.
 */
int swa_watchdog_selftest(int limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SWA_B300_H */
