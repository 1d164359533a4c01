/*
 * fa.h -- C ABI of the GB300 (sm_103a) fused exact-attention library.
 *
 * The library computes exact scaled-dot-product attention
 *     O = softmax(scale * Q K^T) V
 * as one fused kernel per call: Q, K, V are tiled, the scores S and the
 * probabilities P never reach global memory, and an online softmax (running
 * row max m and denominator l, the partial O rescaled when the max moves) is
 * kept per query row. This is the algorithm of "Lesson 1: FlashAttention core
 * idea" §3-§4 and of "FlashAttention and Triton" §19.4-§19.6. The backward
 * pass keeps only one number per query row from the forward pass (the
 * log-sum-exp, "Lesson 1" §5) and recomputes S and P tile by tile.
 *
 * Conventions shared by every entry point
 *  - Tensors are dense, contiguous, row-major [B, H, N, d] (d fastest);
 *    per-row statistics are [B, H, N] float32.
 *  - Every pointer argument is a DEVICE pointer (cudaMalloc / PyTorch CUDA
 *    memory on the current device) unless stated otherwise. The caller owns
 *    all buffers and the stream; the library allocates no device memory and
 *    keeps no pointer after the call returns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Work is enqueued asynchronously; FA_OK means "validated and
 *    launched", not "finished".
 *  - No call throws; errors are returned as fa_status. Arguments are validated
 *    before anything is launched: on any error nothing is enqueued.
 *  - Attention is non-causal, without mask or dropout, unless an _ex or
 *    _varlen entry point is given FA_CAUSAL.
 *
 * dtypes and head sizes
 *  - FA_BF16: bf16 Q/K/V/O/dO/dQ/dK/dV, float32 accumulation, d in {64, 128}.
 *    Runs on the tcgen05 tensor cores. Pointers 16-byte aligned.
 *  - FA_F32 : float32 everything, 1 <= d <= 128, CUDA-core FFMA arithmetic.
 *    Pointers 4-byte aligned.
 *  - Any N >= 1 (ragged last tiles are masked), B >= 1, H >= 1,
 *    B*H*N*d < 2^31 elements per tensor.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, non-positive size, bad scale, small workspace */
  FA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. bf16 with d not in {64,128}) */
  FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a launch failed */
  FA_ERR_TIMEOUT = 4      /* a kernel gave up on a bounded wait (reported by fa_check_device_status) */
} fa_status;

typedef enum { FA_F32 = 0, FA_BF16 = 1 } fa_dtype;

/*
 * Forward pass.  "Lesson 1" §4 (tiled forward, query tiles outer, key/value
 * tiles inner, online softmax, O_i / l_i at the end).
 *   Q, K, V : [B,H,N,d] inputs, dtype `dt`.
 *   O       : [B,H,N,d] output, dtype `dt`.
 *   LSE     : [B,H,N] float32 output, LSE = m + ln(l) of the scaled scores
 *             scale * q.k (natural log). The backward pass consumes it.
 *   scale   : finite, > 0 (the pages use 1/sqrt(d)).
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED (before launch), FA_ERR_CUDA.
 */
fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                 int B, int H, int N, int d, float scale, fa_dtype dt, void* stream);

/* Flags of the _ex and _varlen entry points. */
#define FA_CAUSAL 1 /* query row r attends to keys c <= r of its own sequence */
/* Backward stages (fa_bwd_ex / fa_bwd_varlen); no stage bit = all three, in order. */
#define FA_STAGE_PREPROCESS (1 << 8)
#define FA_STAGE_MAIN (2 << 8)
#define FA_STAGE_DQ_CONVERT (4 << 8)
#define FA_STAGE_MASK (7 << 8)

/*
 * fa_fwd with flags: 0 or FA_CAUSAL. Causal attention is not on the source
 * pages; it is the plainest adjacent variant of the definition for
 * self-attention: row r of softmax(scale * Q K^T) is taken over keys
 * c <= r only (the others get weight 0), O and LSE defined over those keys.
 * Query tiles skip key tiles past their diagonal. Errors: as fa_fwd, plus
 * FA_ERR_INVALID_ARG for unknown flags.
 */
fa_status fa_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE,
                    int B, int H, int N, int d, float scale, int flags, fa_dtype dt, void* stream);

/*
 * Bytes of device scratch with which fa_fwd_ws shortens this problem's
 * forward on the CURRENT device; 0 when it gains nothing (or on invalid
 * arguments). Only bf16, non-causal problems are split.
 */
size_t fa_fwd_workspace_bytes(int B, int H, int N, int d, int flags, fa_dtype dt);

/*
 * The schedule fa_fwd_ws uses: *n_full units (batch*head, 256-query block)
 * run whole, then *n_tail units run as *splits key ranges each (*splits = 1,
 * *n_tail = 0: nothing split). resident_ctas > 0 plans for a GPU running
 * that many forward CTAs at once (host only, no GPU needed); 0 plans for the
 * current device. The rule: with W CTAs at once and U units, the U mod W
 * units of the last wave are split into min(W / (U mod W), 4, key tiles / 4)
 * ranges when that is at least 2 and U >= W (bf16, non-causal only).
 * bf16 d = 64 problems that run on the four-query-tile kernel (causal or
 * not, B*H*ceil(N/512) >= 3/4 of W) are never split.
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED (as fa_fwd_ex).
 */
fa_status fa_fwd_plan(int B, int H, int N, int d, int flags, fa_dtype dt, int resident_ctas,
                      int* n_full, int* n_tail, int* splits);

/*
 * fa_fwd_ex with scratch for the tail of the schedule. The forward runs one
 * CTA per (batch*head, 256-query block) unit, one CTA per SM; when the last
 * wave of CTAs is only partly filled, its units are split into 2-4 key
 * ranges, each range runs as a CTA of its own and leaves a partial result in
 * the scratch, and a second kernel on the same stream combines the parts by
 * their maxima and sums ("Lesson 1: FlashAttention core idea" §3). O and LSE
 * are the same attention (other rounding order within fp32).
 *   workspace       : device scratch of >= fa_fwd_workspace_bytes() bytes,
 *                     256-byte aligned, contents on entry irrelevant, used by
 *                     one call at a time (stream-ordered); NULL (or a
 *                     problem that needs none) runs the plain schedule.
 * Errors: as fa_fwd_ex, plus FA_ERR_INVALID_ARG for a non-NULL workspace
 * that is too small or misaligned.
 */
fa_status fa_fwd_ws(const void* Q, const void* K, const void* V, void* O, float* LSE,
                    void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                    float scale, int flags, fa_dtype dt, void* stream);

/*
 * Variable-length batch (packed layout, no padding): B sequences of
 * different lengths, sequence b holding rows cu_seqlens[b] ..
 * cu_seqlens[b+1]-1 of the packed tensors. Each sequence is attended to
 * separately (keys of other sequences get weight 0); with FA_CAUSAL row r
 * of a sequence sees its keys 0..r.
 *   Q, K, V, O : [total, H, d] (rows of all sequences back to back, then
 *                heads, d fastest), dtype `dt`.
 *   LSE        : [H, total] float32 output.
 *   cu_seqlens : DEVICE int32 [B+1], cu_seqlens[0] = 0, non-decreasing,
 *                cu_seqlens[B] = total; every length <= max_seqlen <= total
 *                (max_seqlen sizes the grid). The kernels check each pair:
 *                a sequence whose offsets break these rules is skipped
 *                (nothing of it is read or written) and fa_check_device_status
 *                then returns FA_ERR_INVALID_ARG.
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED (as fa_fwd; H*total*d <
 * 2^31, B*H <= 65535), FA_ERR_CUDA.
 */
fa_status fa_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE,
                        const int* cu_seqlens, int B, int H, int total, int max_seqlen, int d,
                        float scale, int flags, fa_dtype dt, void* stream);

/*
 * Bytes of device scratch that fa_bwd needs for this problem on the CURRENT
 * device (0 on invalid arguments). The caller allocates it; its contents on
 * entry do not matter. Holds the fp32 dQ accumulator, per-row statistics
 * derived from D = rowsum(dO o O) and the LSE, the main kernel's unit
 * counter and, when the schedule splits its tail (fa_bwd_plan), the split
 * units' fp32 partial dK and dV.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d, fa_dtype dt);

/*
 * The schedule of the bf16 backward's main kernel for this problem (no GPU
 * work). Its work items are (batch*head, 128-key tile) units, taken by a
 * persistent grid of one CTA per SM (non-causal: item w by CTA w mod W, in
 * order);
 * when the last round of items fills at most half of the SMs, its *n_tail
 * units run as *splits ranges of query tiles each, one item per range, and the dQ-convert
 * stage adds their partial dK and dV up ("Lesson 1: FlashAttention core
 * idea" §5: dK_j and dV_j are sums over the query tiles). *n_full units run
 * whole (*splits = 1, *n_tail = 0: nothing split). The rule, with W CTAs at
 * once and U units: splits = min(W / (U mod W), 4, query tiles / 4) when that
 * is at least 2 and U >= W; bf16, fixed length, non-causal only. The partial
 * sums are part of fa_bwd_workspace_bytes().
 *   resident_ctas : W; 0 plans for the current device.
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED (as fa_bwd_ex).
 */
fa_status fa_bwd_plan(int B, int H, int N, int d, int flags, fa_dtype dt, int resident_ctas,
                      int* n_full, int* n_tail, int* splits);

/*
 * Backward pass with recomputation.  "Lesson 1" §5: with P rebuilt from the
 * saved statistics, dV = P^T dO, dP = dO V^T,
 * dS = P o (dP - rowsum(dO o O)) * scale, dQ = dS K, dK = dS^T Q.
 * (rowsum(dP o P) over a full row equals rowsum(dO o O) because O = P V.)
 *   Q, K, V, O, dO : [B,H,N,d] inputs, dtype `dt` (O from fa_fwd).
 *   LSE            : [B,H,N] float32 from fa_fwd.
 *   dQ, dK, dV     : [B,H,N,d] outputs, dtype `dt`.
 *   workspace      : device scratch of >= fa_bwd_workspace_bytes() bytes,
 *                    256-byte aligned, not used by another call in flight.
 * Errors: as fa_fwd, plus FA_ERR_INVALID_ARG when the workspace is too small.
 */
fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV, void* workspace,
                 size_t workspace_bytes, int B, int H, int N, int d, float scale, fa_dtype dt,
                 void* stream);

/*
 * One stage of fa_bwd, for callers that schedule or time the stages
 * separately. Same arguments and validation as fa_bwd, plus `stage`:
 *   FA_BWD_PREPROCESS (0): per-row statistics from D = rowsum(dO o O) and
 *                          the LSE into the workspace; zero the workspace's
 *                          dQ accumulator and (bf16) the main stage's unit
 *                          counter.
 *   FA_BWD_MAIN       (1): recompute P tile by tile; write dK, dV (the
 *                          split units of fa_bwd_plan: partial sums into the
 *                          workspace); add dQ into the workspace accumulator
 *                          (for bf16 without the softmax scale). Needs stage
 *                          0 done since the last main stage on this
 *                          workspace (a causal bf16 problem takes its units
 *                          from that counter).
 *   FA_BWD_DQ_CONVERT (2): workspace dQ accumulator -> dQ in dtype `dt`
 *                          (bf16: the scale is applied here), and the split
 *                          units' partial dK, dV added up into dK, dV.
 *                          Needs stage 1.
 * Stages run in that order on one workspace; fa_bwd == stages 0, 1, 2.
 * Errors: as fa_bwd, plus FA_ERR_INVALID_ARG for an unknown stage.
 */
typedef enum { FA_BWD_PREPROCESS = 0, FA_BWD_MAIN = 1, FA_BWD_DQ_CONVERT = 2 } fa_bwd_stage_id;

/*
 * fa_bwd with flags: FA_CAUSAL and/or stage bits (FA_STAGE_PREPROCESS,
 * FA_STAGE_MAIN, FA_STAGE_DQ_CONVERT; none = all three). The workspace is the
 * same as fa_bwd's. Pass the flags given to fa_fwd_ex. With FA_CAUSAL the
 * gradients are those of the causal definition: P is zero above the
 * diagonal, so key tiles skip the query tiles before their diagonal.
 * Errors: as fa_bwd, plus FA_ERR_INVALID_ARG for unknown flags.
 */
fa_status fa_bwd_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                    const float* LSE, void* dQ, void* dK, void* dV, void* workspace,
                    size_t workspace_bytes, int B, int H, int N, int d, float scale, int flags,
                    fa_dtype dt, void* stream);

/* Scratch bytes for fa_bwd_varlen (0 on invalid sizes). */
size_t fa_bwd_varlen_workspace_bytes(int B, int H, int total, int max_seqlen, int d, fa_dtype dt);

/*
 * Backward pass of fa_fwd_varlen: same packed layout ([total, H, d] tensors,
 * LSE [H, total], device cu_seqlens), flags and stage bits as fa_bwd_ex,
 * workspace of >= fa_bwd_varlen_workspace_bytes() bytes, 256-byte aligned.
 * Errors: as fa_fwd_varlen, plus FA_ERR_INVALID_ARG for a small workspace.
 */
fa_status fa_bwd_varlen(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                        const float* LSE, void* dQ, void* dK, void* dV, const int* cu_seqlens,
                        void* workspace, size_t workspace_bytes, int B, int H, int total,
                        int max_seqlen, int d, float scale, int flags, fa_dtype dt, void* stream);

fa_status fa_bwd_stage(int stage, const void* Q, const void* K, const void* V, const void* O,
                       const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                       void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                       float scale, fa_dtype dt, void* stream);

/*
 * Fused row softmax: Y[r, :] = softmax(scale * X[r, :]) for each of `rows`
 * rows of `cols` elements. The fusion example of "FlashAttention and Triton"
 * §19.11: one pass per row (a ragged tail reads as -inf), max, exp, sum and
 * divide without intermediate arrays, so each element is read and written
 * once. X, Y: dense row-major [rows, cols], dtype `dt` (fp32 or bf16, the
 * arithmetic in fp32); they may alias (in place). 1 <= cols <= 32768,
 * rows >= 1, rows * cols < 2^31, scale finite and > 0.
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED (cols > 32768), FA_ERR_CUDA.
 */
fa_status fa_softmax_rows(const void* X, void* Y, int rows, int cols, float scale, fa_dtype dt,
                          void* stream);

/*
 * KV-cache decode: attention of Nq new queries per head against Nk cached
 * keys and values, O = softmax(scale * Q K^T) V and LSE = ln sum exp(scale *
 * Q K^T) per query row, every query seeing every key (no mask). The use case
 * is the inference remark of "Interview Q15: FlashAttention" (decoding with a
 * KV cache). The keys are cut into contiguous splits processed in parallel,
 * each with the online softmax of "Lesson 1: FlashAttention core idea" §3;
 * the split results (normalised output and log-sum-exp) are merged with the
 * same (m, l) rule by a second kernel. Nothing of size Nq x Nk reaches
 * global memory.
 *   Q, O : [B,H,Nq,d] bf16 (for grouped-query attention pass the G query
 *          heads that share one K/V head as Nq = G rows).
 *   K, V : [B,H,Nk,d] bf16, the cache; only the first Nk rows are read.
 *   LSE  : [B,H,Nq] float32 output (natural log, as fa_fwd).
 *   workspace : device scratch of >= fa_decode_workspace_bytes() bytes,
 *          256-byte aligned, not used by another call in flight; contents on
 *          entry do not matter (split outputs and log-sum-exps, fp32).
 *   dt   : FA_BF16 only; d in {64, 128}; 1 <= Nq <= 16; 1 <= Nk <= 2^30;
 *          B*H <= 65535. Q, K, V, O 16-byte aligned, LSE 4-byte aligned.
 * One query per head runs on CUDA cores (bandwidth-bound); 2..16 queries
 * run both products on the tensor cores with the queries padded to 16.
 * Errors: FA_ERR_INVALID_ARG (pointers, sizes, scale, small workspace),
 * FA_ERR_UNSUPPORTED (FA_F32, d, Nq > 16), FA_ERR_CUDA.
 */
fa_status fa_decode(const void* Q, const void* K, const void* V, void* O, float* LSE,
                    void* workspace, size_t workspace_bytes, int B, int H, int Nq, int Nk, int d,
                    float scale, fa_dtype dt, void* stream);

/*
 * Bytes of scratch fa_decode needs for this problem on the CURRENT device
 * (the split count depends on its SM count); 0 on invalid arguments or a
 * failed device query.
 */
size_t fa_decode_workspace_bytes(int B, int H, int Nq, int Nk, int d, fa_dtype dt);

/*
 * The split plan fa_decode uses: *splits key ranges of *keys_per_split keys
 * (a multiple of 64; the last range may be shorter), chosen to fill whole
 * waves of resident CTAs. resident_ctas > 0 plans for a GPU that holds that
 * many decode CTAs at once (no device access, for tests and capacity
 * planning); resident_ctas == 0 queries the current device. Returns
 * FA_ERR_INVALID_ARG on bad sizes or null outputs, FA_ERR_CUDA if the device
 * query fails.
 */
fa_status fa_decode_plan(int B, int H, int Nq, int Nk, int d, int resident_ctas, int* splits,
                         int* keys_per_split);

/*
 * fa_bwd without a caller-provided workspace, for callers that cannot
 * allocate device memory (for example code running inside a host application
 * that owns all device memory through its own pool, or a serving path where
 * cudaMalloc is not allowed). The paper has no counterpart to this entry point:
 * it is a deployment convenience around fa_bwd.
 * Same arguments, results and errors as fa_bwd, minus the workspace. The
 * scratch is one library-owned device array of
 * FA_BWD_NOALLOC_MAX_WORKSPACE_BYTES per device, held until process exit;
 * problems needing more (fa_bwd_workspace_bytes) return FA_ERR_UNSUPPORTED
 * without launching. All calls on a device share that array: calls whose
 * kernels may overlap on the GPU race and must be ordered by the caller. The
 * first call on each device looks up the array's address; make it before any
 * stream capture. Allocates nothing.
 */
#define FA_BWD_NOALLOC_MAX_WORKSPACE_BYTES ((size_t)32 << 20)

fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                         int B, int H, int N, int d, float scale, fa_dtype dt, void* stream);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word on the current device. Returns FA_ERR_TIMEOUT if any kernel launched
 * since the last check abandoned a bounded wait (its outputs are then
 * undefined), FA_ERR_INVALID_ARG if a variable-length call met inconsistent
 * cu_seqlens (the sequences concerned were skipped), FA_ERR_CUDA if the
 * stream reports an error, FA_OK otherwise.
 */
fa_status fa_check_device_status(void* stream);

/*
 * Test hook for the bounded-wait machinery: launches one block that waits on
 * a shared-memory barrier nothing will ever arrive at, giving up after
 * `limit_ns` nanoseconds (clamped to [1e3, 2e9]) and recording FA_ERR_TIMEOUT
 * in the device status word, exactly as the attention kernels do. Lets a test
 * observe the timeout path without hanging or faulting the GPU.
 */
fa_status fa_debug_timeout_probe(long long limit_ns, void* stream);

/*
 * Test hooks for the attention kernels' own abort path (bf16 only). Same
 * arguments, layout and ownership as fa_fwd / fa_bwd (dtype bf16, no causal
 * mask), plus:
 *   skip_tile  the forward's producer skips the load of key tile `skip_tile`
 *              of every CTA; the backward's producer skips the Q tile of
 *              query iteration `skip_tile` of every CTA (a CTA of the
 *              persistent grid counts its iterations over all the units it
 *              walks, in order). Neither the copy nor
 *              its expected-bytes arrival is issued, so no copy is left in
 *              flight; the consumers' bounded waits on that tile run out.
 *              Must be in [1, ceil(N / 128) - 1], else FA_ERR_INVALID_ARG.
 *   limit_ns   every bounded wait of these launches gives up after this many
 *              nanoseconds (clamped to [1e3, 2e9]).
 * Each CTA then records FA_ERR_TIMEOUT in the device status word, waits for
 * the copies and products it issued, frees its tensor memory and exits; the
 * outputs are undefined. fa_check_device_status reports (and clears) the
 * timeout, and the context stays usable for ordinary calls. Not for
 * production use: the pages have no counterpart; this exercises the bounded
 * waits every kernel here carries.
 */
fa_status fa_debug_fwd_skip_load(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                 int B, int H, int N, int d, float scale, int skip_tile,
                                 long long limit_ns, void* stream);
fa_status fa_debug_bwd_skip_load(const void* Q, const void* K, const void* V, const void* O,
                                 const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                                 void* workspace, size_t workspace_bytes, int B, int H, int N,
                                 int d, float scale, int skip_tile, long long limit_ns,
                                 void* stream);
/*
 * fa_debug_bwd_skip_load with flags: FA_CAUSAL runs the causal backward,
 * whose persistent CTAs take their units from the device counter and pass
 * them on through the shared-memory item ring (the ring's bounded waits then
 * run out too). The workspace must hold fa_bwd_workspace_bytes for the
 * problem. Errors: as fa_debug_bwd_skip_load, plus FA_ERR_INVALID_ARG for
 * flags other than 0 and FA_CAUSAL.
 */
fa_status fa_debug_bwd_skip_load_ex(const void* Q, const void* K, const void* V, const void* O,
                                    const void* dO, const float* LSE, void* dQ, void* dK,
                                    void* dV, void* workspace, size_t workspace_bytes, int B,
                                    int H, int N, int d, float scale, int flags, int skip_tile,
                                    long long limit_ns, void* stream);

/* Static, NUL-terminated description of a status code. */
const char* fa_status_string(fa_status s);

/* Library ABI version (major * 100 + minor). */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
