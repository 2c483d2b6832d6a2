/*
 * csa.h -- C ABI of the B300 (sm_103a) hybrid long-context attention library.
 *
 * The operations are the steps of DeepSeek-V4's hybrid attention as described
 * in "DeepSeek V4 技术解读" (takeshell.com):
 *   §2.1 CSA  -- compress every m tokens' KV into one entry, score the entries
 *                with the Lightning Indexer, keep the top-k, attend over them;
 *   §2.2 HCA  -- compress at m' = 128, attend densely over all entries;
 *   §2.3      -- the first layers use sliding-window attention;
 *   §五       -- FP4 (E2M1) indexer keys are widened to FP8 (E4M3).
 *
 * Conventions shared by every call:
 *   - All tensors are dense row-major device buffers owned by the caller,
 *     16-byte aligned (else CSA_ERR_ALIGNMENT).  The library allocates no
 *     device memory; calls that need scratch take a caller-owned workspace
 *     whose size the matching *_workspace_size() query returns.
 *   - Every call is asynchronous on the given stream (NULL = legacy default
 *     stream).  Argument errors are returned before anything is launched;
 *     a failed launch returns CSA_ERR_CUDA.  Messages: csa_last_error().
 *   - Kernels never trap.  A device-side wait that exceeds its time limit, or
 *     a bounds violation, sets a per-device status word that
 *     csa_device_status() reports (CSA_ERR_TIMEOUT / CSA_ERR_DEVICE).
 *   - Results are deterministic and batch-invariant: no floating-point
 *     atomics, fixed reduction orders ("DeepSeek V4 技术解读" §6.2).
 *   - Shapes use: B batch, n raw tokens, m compression ratio,
 *     N_c = floor(n / m) closed compressed entries, H / d attention heads and
 *     head dim, H_I / d_I indexer heads and head dim, k top-k.  The query at
 *     absolute position t sees entry j iff (j + 1) * m - 1 <= t, i.e. the
 *     nv(t) = min(floor((t + 1) / m), N_c) first entries.
 *   - Attention uses one KV head shared by all H query heads (H_kv = 1); the
 *     attention calls also take H_kv > 1 KV heads (GQA / MHA readings).
 */
#ifndef CSA_H
#define CSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* csa_stream_t;

typedef enum {
    CSA_OK = 0,
    CSA_ERR_INVALID_ARG = 1,   /* bad size, pointer or dtype combination       */
    CSA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (shape / dtype)     */
    CSA_ERR_ALIGNMENT = 3,     /* a pointer is not 16-byte aligned              */
    CSA_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required    */
    CSA_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed          */
    CSA_ERR_TIMEOUT = 6,       /* a device wait exceeded its limit              */
    CSA_ERR_DEVICE = 7         /* a device-side bounds check failed             */
} csa_status_t;

typedef enum {
    CSA_F32 = 0,
    CSA_BF16 = 1,
    CSA_E4M3 = 2,   /* OCP FP8 E4M3 ("fn": max 448, no inf) codes, 1 byte each */
    CSA_E2M1 = 3    /* OCP FP4 E2M1 codes, 2 per byte, element 2i in the low nibble */
} csa_dtype_t;

/* ---------------------------------------------------------------------------
 * csa_compress -- KV compression ("DeepSeek V4 技术解读" §2.1 KV Cache 压缩,
 * §2.2).  For each of n_streams streams (K, V, indexer K, ...) sharing one
 * logits tensor:
 *     out[b, j, :] = sum_{i<m} w[b, j, i] * x[b, j*m + i, :],
 *     w[b, j, :]   = softmax(logits[b, j*m .. j*m + m - 1]),
 * for j < N_c (a trailing partial block is dropped).  fp32 accumulation.
 *   logits      device, fp32 [B, n].
 *   x[s]        device, [B, n, dim[s]] in x_dtype[s] (CSA_F32 or CSA_BF16).
 *   out[s]      device, [B, N_c, dim[s]] in out_dtype[s]:
 *                 CSA_F32 / CSA_BF16  rounded to nearest even;
 *                 CSA_E4M3  codes [B, N_c, dim], out_scale[s] fp32 [B, N_c]:
 *                           scale = amax / 448, code = E4M3(x * (448 / amax)),
 *                           an all-zero row gets scale 1;
 *                 CSA_E2M1  packed codes [B, N_c, dim / 2], out_scale[s] E4M3
 *                           block scales [B, N_c, dim / 32]:
 *                           sc = E4M3(amax_32 / 6) (at least the smallest
 *                           positive E4M3), code = E2M1(x / sc).
 *   out_scale   host array of n_streams device pointers (entries may be NULL
 *               for unscaled outputs); the array itself may be NULL.
 *   x, x_dtype, dim, out, out_dtype: host arrays of n_streams entries.
 * Requirements: 1 <= n_streams <= 4, m >= 1, dim[s] a power of two in
 * [8, 256] (at least 32 for CSA_E2M1); otherwise CSA_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------- */
csa_status_t csa_compress(int B, int n, int m, const float* logits, int n_streams,
                          const void* const* x, const csa_dtype_t* x_dtype, const int* dim,
                          void* const* out, const csa_dtype_t* out_dtype,
                          void* const* out_scale, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_compress_per_channel -- the per-channel variant reading of "weighted
 * aggregation" ("DeepSeek V4 技术解读" §2.1 KV Cache 压缩): every channel has
 * its own logit per token, and
 *     out[b, j, c] = sum_{i<m} softmax_i(logits[s][b, j*m + i, c]) x[b, j*m + i, c].
 *   logits   host array of n_streams device pointers, fp32 [B, n, dim[s]].
 *   Other arguments, outputs and requirements as in csa_compress.
 * ------------------------------------------------------------------------- */
csa_status_t csa_compress_per_channel(int B, int n, int m, int n_streams, const float* const* logits,
                                      const void* const* x, const csa_dtype_t* x_dtype, const int* dim,
                                      void* const* out, const csa_dtype_t* out_dtype,
                                      void* const* out_scale, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_index_scores -- Lightning Indexer scores ("DeepSeek V4 技术解读" §2.1,
 * 64 indexer heads x 128; §五 for the FP4 keys):
 *     s[b, i, j] = sum_h sq[b,i,h] * sk[b,j] * < q[b,i,h,:], k[b,j,:] >
 * for j < nv(q_pos0 + i); entries j >= nv are left unwritten.
 *   q_idx    device [B, n_q, H_I, d_I]: CSA_F32, CSA_BF16, or CSA_E4M3 with
 *            q_scale fp32 [B, n_q, H_I] (NULL means 1).
 *   k_idx    device [B, N_c, d_I]: CSA_F32 / CSA_BF16 (k_scale NULL),
 *            CSA_E4M3 with k_scale fp32 [B, N_c], or CSA_E2M1 packed
 *            [B, N_c, d_I / 2] with k_scale E4M3 block scales
 *            [B, N_c, d_I / 32].  E2M1 keys are first widened to E4M3 per row:
 *            S = 2^(floor(log2 max_b sc_b) - 5), x8 = E4M3(e * sc_b / S),
 *            sk = S (exact unless e * sc_b / S falls off the E4M3 grid).
 *   scores   device [B, n_q, N_c] in score_dtype: CSA_F32, or CSA_BF16 (the
 *            fp32 score rounded to nearest even; the score storage precision
 *            of "DeepSeek-V4 点评总结", FP4 量化感知训练: half the score
 *            traffic, at a recall cost the tests measure).
 *   head_weight, relu  the weighted / ReLU variant reading of the indexer's
 *            "similarity" (§2.1): head_weight device fp32 [B, n_q, H_I] (or
 *            NULL: weight 1) and relu != 0 give
 *            s = sk * sum_h w(t,h) * sq(t,h) * max(<q(t,h), k(j)>, 0).
 *            NULL and 0 give the plain score above.
 * Precision pairs: (F32, F32) on CUDA cores; (BF16, BF16) and
 * (E4M3, E4M3 | E2M1) on tcgen05 tensor cores with fp32 accumulation, which
 * require H_I = 64 and d_I = 128.
 * ------------------------------------------------------------------------- */
size_t csa_index_scores_workspace_size(int B, int N_c, int d_I, csa_dtype_t k_dtype);
csa_status_t csa_index_scores(int B, int n_q, int64_t q_pos0, int m, int N_c, int H_I, int d_I,
                              const void* q_idx, csa_dtype_t q_dtype, const float* q_scale,
                              const void* k_idx, csa_dtype_t k_dtype, const void* k_scale,
                              const float* head_weight, int relu,
                              void* scores, csa_dtype_t score_dtype, void* workspace,
                              size_t workspace_bytes, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_topk_select -- top-k selection ("DeepSeek V4 技术解读" §2.1: keep the k
 * best-scoring compressed entries).  Row (b, i) ranks its nv(q_pos0 + i)
 * visible scores by (score descending, index ascending), -0 equal to +0, and
 * writes the first min(k, nv) indices in ascending order, padded with -1.
 * Exact radix selection on the bit patterns of the stored scores.
 *   scores   device [B, n_q, N_c] in score_dtype (CSA_F32 or CSA_BF16; the
 *            ranking is that of the stored values, so bf16 ties go to the
 *            smaller index);  topk  device int32 [B, n_q, k].
 * Requirements: 1 <= k <= 4096, N_c <= 524288, and B * n_q (times
 * ceil(N_c / 32768) for rows longer than 32,768 entries) at most INT_MAX;
 * otherwise CSA_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------- */
size_t csa_topk_select_workspace_size(int B, int n_q, int N_c, int k);
csa_status_t csa_topk_select(int B, int n_q, int64_t q_pos0, int m, int N_c, int k,
                             const void* scores, csa_dtype_t score_dtype, int32_t* topk,
                             void* workspace, size_t workspace_bytes, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_topk_select_noalloc -- the same selection as csa_topk_select, for
 * callers that cannot allocate device memory: a plugin inside another
 * runtime that owns all of the device's memory and passes this library only
 * its input and output buffers, or a latency-critical path where a
 * cudaMalloc, which can synchronise the device, is not acceptable.  The
 * method's description has no counterpart of this call; it is an addition of
 * this library.
 *   Arguments and results as in csa_topk_select with fp32 scores, without
 *   the workspace.
 *   Scratch: a fixed device array of CSA_TOPK_NOALLOC_SCRATCH_BYTES (4 MiB)
 *   inside the library.  Rows longer than 32,768 entries need 8 * max(8192,
 *   4k) bytes of it each, plus a few bytes (csa_topk_select_workspace_size
 *   reports the need): with k = 1024, up to 63 such rows fit in one call --
 *   e.g. 63 decode queries over 262,144 entries; shorter rows need none.  Larger selections return CSA_ERR_WORKSPACE and
 *   launch nothing.  Every GPU that loads the library holds the array until
 *   the process exits.
 *   The call allocates nothing.  Its first call on a device looks up the
 *   array's device address (cudaGetSymbolAddress) with that device current;
 *   make that first call before any stream capture.  All calls on a device
 *   share the one array and it keeps the last call's contents, so calls that
 *   overlap on the GPU (several streams or host threads) race: serialise them.
 * ------------------------------------------------------------------------- */
#define CSA_TOPK_NOALLOC_SCRATCH_BYTES (4u << 20)
csa_status_t csa_topk_select_noalloc(int B, int n_q, int64_t q_pos0, int m, int N_c, int k,
                                     const float* scores, int32_t* topk, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_index_topk -- scores and selection in one call (csa_index_scores then
 * csa_topk_select), processing the queries in chunks so that the score
 * buffer (score_dtype, in the workspace) stays within 256 MB.  Arguments as
 * above.  For fewer than four queries a sequence over rows longer than
 * 32,768 entries (decode), the tensor-core indexer also writes the largest
 * score of every 32 consecutive entries, and the selection takes its
 * collection threshold from them (the k-th largest has at least k entries at
 * or above it) instead of from a sample of the row, and reads only the runs
 * of 32 whose largest score reaches it.
 * ------------------------------------------------------------------------- */
size_t csa_index_topk_workspace_size(int B, int n_q, int N_c, int H_I, int d_I, int k,
                                     csa_dtype_t k_dtype, csa_dtype_t score_dtype);
csa_status_t csa_index_topk(int B, int n_q, int64_t q_pos0, int m, int N_c, int H_I, int d_I,
                            int k, const void* q_idx, csa_dtype_t q_dtype, const float* q_scale,
                            const void* k_idx, csa_dtype_t k_dtype, const void* k_scale,
                            const float* head_weight, int relu,
                            csa_dtype_t score_dtype, int32_t* topk, void* workspace,
                            size_t workspace_bytes, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_index_topk_varlen -- csa_index_topk for sequences of different lengths
 * held on the device: query i of sequence b sits at position
 * lens[b] - n_q + i (lens: device int64 [B], the tokens of each sequence
 * including its n_q queries -- the counts csa_decode_append keeps).  N_c is
 * the caches' capacity (entries per sequence); sequence b sees its first
 * min(floor((lens[b] - n_q + i + 1) / m), N_c) entries (none where that
 * position is negative: lens[b] < n_q).  Other arguments,
 * outputs and the workspace as in csa_index_topk.
 * ------------------------------------------------------------------------- */
csa_status_t csa_index_topk_varlen(int B, int n_q, const int64_t* lens, int m, int N_c, int H_I, int d_I,
                                   int k, const void* q_idx, csa_dtype_t q_dtype, const float* q_scale,
                                   const void* k_idx, csa_dtype_t k_dtype, const void* k_scale,
                                   const float* head_weight, int relu,
                                   csa_dtype_t score_dtype, int32_t* topk, void* workspace,
                                   size_t workspace_bytes, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_decode_append -- streaming decode state: the KV-cache compression of
 * "DeepSeek V4 技术解读" §2.1 (every m tokens merged into one entry) applied
 * one generated token at a time.  For every sequence b (t = lens[b] tokens
 * so far): the new token (its logit, K, V and indexer-K rows) is written to
 * slot t % m of the sequence's open block (the stage buffers), lens[b]
 * becomes t + 1, and when t + 1 is a multiple of m the block is compressed
 * -- softmax of its m logits, fp32 sums in token order, the quantising
 * epilogue of csa_compress -- into entry (t + 1) / m - 1 of the caches.
 *   logit_new fp32 [B]; k_new, v_new [B, d]; ik_new [B, d_I]  (x_dtype:
 *             CSA_F32 or CSA_BF16), device;
 *   stage_logits fp32 [B, m]; stage_k, stage_v [B, m, d]; stage_ik
 *             [B, m, d_I] (x_dtype): the open blocks, caller-owned, device;
 *   lens      device int64 [B], advanced by one;
 *   k_c, v_c  device [B, N_cap, d] in kv_dtype (CSA_F32 or CSA_BF16);
 *   ik_c, ik_scale  indexer-key cache [B, N_cap, d_I] in ik_dtype: CSA_F32 /
 *             CSA_BF16 (ik_scale unused), CSA_E4M3 (ik_scale fp32 [B, N_cap]),
 *             or CSA_E2M1 (packed [B, N_cap, d_I / 2], ik_scale E4M3
 *             [B, N_cap, d_I / 32]).
 * Requirements: 1 <= m <= 128, d and d_I <= 256, d_I even (a multiple of 32
 * for E2M1).  A block closing past N_cap entries is not written, and a
 * negative lens[b] leaves sequence b untouched; both flag CSA_ERR_DEVICE in
 * the status word.  Deterministic; sequences are
 * independent (one CTA each).
 * ------------------------------------------------------------------------- */
csa_status_t csa_decode_append(int B, int m, int d, int d_I, int64_t N_cap, const float* logit_new,
                               const void* k_new, const void* v_new, const void* ik_new, csa_dtype_t x_dtype,
                               float* stage_logits, void* stage_k, void* stage_v, void* stage_ik,
                               int64_t* lens, void* k_c, void* v_c, csa_dtype_t kv_dtype, void* ik_c,
                               csa_dtype_t ik_dtype, void* ik_scale, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_sparse_attn -- CSA core attention ("DeepSeek V4 技术解读" §2.1 Core
 * Attention: full attention over only the k selected entries):
 *     o[b,i,h,:] = sum_{j in topk[b,i,:], j >= 0} softmax_j(scale * <q, k_c[b,j]>) v_c[b,j,:]
 *     lse[b,i,h] = log sum_j exp(scale * <q, k_c[b,j]>)      (natural log)
 * An empty selection gives o = 0 and lse = -inf.
 *   q      device [B, n_q, H, d];  k_c, v_c  device [B, N_c, H_kv, d];  all
 *          in dtype (CSA_F32 or CSA_BF16);  out  device [B, n_q, H, d] in dtype;
 *   H_kv   KV heads: 1 is the shared head of the MLA reading (the spec's);
 *          H_kv > 1 (dividing H, H / H_kv a power of two <= 128) are the GQA
 *          and MHA variant readings, query head h reading KV head
 *          h / (H / H_kv);
 *   topk   device int32 [B, n_q, k], entries in [0, N_c) or -1;
 *   lse    device fp32 [B, n_q, H] or NULL.
 * Requirements: d in {64, 128}, H in {8, 16, 32, 64, 128} for H_kv = 1,
 * scale > 0 and finite (else CSA_ERR_INVALID_ARG).  Indices outside
 * [-1, N_c) are skipped and flagged in the device status word.
 * Precision: BF16 with one KV head, d = 128 and H in {64, 128} runs on the
 * tcgen05 tensor cores (the probabilities enter the P.V product rounded to
 * bf16, fp32 accumulation); other shapes, H_kv > 1 and fp32 I/O run on CUDA
 * cores in fp32.
 * ------------------------------------------------------------------------- */
size_t csa_sparse_attn_workspace_size(int B, int n_q, int H, int d, int k);
csa_status_t csa_sparse_attn(int B, int n_q, int H, int H_kv, int d, int N_c, int k, float scale,
                             const void* q, const void* k_c, const void* v_c, csa_dtype_t dtype,
                             const int32_t* topk, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * hca_attn -- HCA dense attention ("DeepSeek V4 技术解读" §2.2): attention of
 * query i (absolute position q_pos0 + i) over all visible compressed entries
 * j < nv(q_pos0 + i), with no selection.  Layouts and output as in
 * csa_sparse_attn.
 * ------------------------------------------------------------------------- */
csa_status_t hca_attn(int B, int n_q, int64_t q_pos0, int m, int N_c, int H, int H_kv, int d, float scale,
                      const void* q, const void* k_c, const void* v_c, csa_dtype_t dtype,
                      void* out, float* lse, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * swa_attn -- sliding-window attention over raw tokens ("DeepSeek V4 技术解读"
 * §2.3): query i at t = q_pos0 + i sees tokens s with t - window < s <= t and
 * s < n_kv.  k, v device [B, n_kv, H_kv, d]; other layouts as in
 * csa_sparse_attn.
 * ------------------------------------------------------------------------- */
csa_status_t swa_attn(int B, int n_q, int64_t q_pos0, int n_kv, int window, int H, int H_kv, int d,
                      float scale, const void* q, const void* k, const void* v,
                      csa_dtype_t dtype, void* out, float* lse, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_device_status -- synchronises the stream, then reads and clears this
 * device's status word: CSA_OK, CSA_ERR_TIMEOUT (a bounded device wait gave
 * up) or CSA_ERR_DEVICE (a device-side bounds check failed).
 *   The status word is ONE word per device, shared by every call of this
 *   library on every stream and host thread of the process: a flag raised by
 *   a kernel on one stream is seen (and cleared) by csa_device_status on any
 *   other stream of the same device.  Callers that run the library on
 *   several streams at once and need per-stream attribution must serialise
 *   the calls they check, or treat a non-OK status as a device-wide event.
 * csa_last_error -- message of the last non-OK status on this host thread.
 * ------------------------------------------------------------------------- */
csa_status_t csa_device_status(csa_stream_t stream);
const char* csa_last_error(void);

/* ---------------------------------------------------------------------------
 * csa_wait_selftest -- exercises the bounded waits every kernel of this
 * library relies on (failure detection without a fault: a device wait that
 * cannot complete gives up, records CSA_ERR_TIMEOUT in the status word and
 * lets its CTA exit, leaving the context usable).  Launches one CTA whose
 * first warp waits on an mbarrier that nothing completes, with a limit of
 * limit_us microseconds (1 .. 2,000,000), and whose second warp waits on
 * another such barrier until the first warp's timeout raises the CTA's abort
 * flag.  No copy, MMA or tensor memory is in flight during the waits.
 *   aborted  device uint32 (16-byte aligned): set to 1 if the second warp was
 *            stopped by the abort flag (well before its own 2 s limit).
 * Returns CSA_OK once launched; csa_device_status() then reports
 * CSA_ERR_TIMEOUT.  The method's description has no counterpart of this call.
 * ------------------------------------------------------------------------- */
csa_status_t csa_wait_selftest(uint32_t limit_us, uint32_t* aborted, csa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA_H */
