/*
 * nsa.h -- C ABI of libnsa.so, the GB300 (sm_103a) native-sparse-attention hot path.
 *
 * Sources, cited by page title and section:
 *   [NOSA-Triton]  "NOSA-1B source walk-through #3: how the Triton kernel speeds up attention"
 *   [NOSA-Parts]   "NOSA-1B core components: how KV-cache offload gives 5.04x decode throughput"
 *   [NSA-Triton]   "DeepSeek NSA sparse attention in practice: optimising training with Triton"
 *   [TileLang-NSA] "TileLang operator development: Native Sparse Attention implementation"
 *
 * Conventions shared by every entry point
 *   - Every tensor argument is caller-owned DEVICE memory, dense row-major in the
 *     layout given, 16-byte aligned.  The library allocates nothing.
 *   - Token-major layouts.  Q and O are [tokens, h, d]; K and V are [tokens, h_kv, d].
 *     A dense batch [B, T, ...] is the packed layout with B sequences of T tokens.
 *     With cu_seqlens (device int32 [n_seqs+1], prefix sums starting at 0) the tokens of
 *     sequence i are rows cu_seqlens[i] .. cu_seqlens[i+1]-1.  Positions t are relative
 *     to the sequence start.
 *   - Grouped-query attention: head hh reads kv-head hh / (h / h_kv)  ([TileLang-NSA]
 *     sec. 2, "head_kv = heads // groups").
 *   - Compressed keys: window `kernel`, step `stride` ([NOSA-Parts] core component 1:
 *     32 and 16).  A sequence of length L has n_c(L) = (L-kernel)/stride + 1 full windows
 *     (0 if L < kernel).  Compressed rows of all sequences are packed one sequence after
 *     another: [sum_i n_c(L_i), h_kv, d].  Compressed key c is causal for query t when
 *     its window has ended: c*stride + kernel - 1 <= t.
 *   - Selection blocks of block_size tokens; a sequence has n_b(L) = ceil(L/block_size).
 *   - scale <= 0 selects 1/sqrt(d).
 *   - Execution is asynchronous on `stream`; no call synchronises the host.
 *   - Errors: argument errors return NSA_ERR_INVALID / NSA_ERR_UNSUPPORTED before any
 *     launch; a failed launch returns NSA_ERR_CUDA.  nsa_last_error() gives a message
 *     (per calling thread).  No C++ exception crosses this interface.  There is no CPU
 *     fallback: a shape the kernels do not cover is rejected.
 */
#ifndef NSA_H_
#define NSA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define NSA_API __attribute__((visibility("default")))
#else
#define NSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NSA_OK = 0,
  NSA_ERR_INVALID = 1,     /* null/misaligned pointer, inconsistent sizes            */
  NSA_ERR_UNSUPPORTED = 2, /* valid arguments outside the shapes the kernels cover   */
  NSA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed                   */
  NSA_ERR_TIMEOUT = 4      /* a device-side bounded wait ran out (nsa_device_status)  */
} nsa_status;

typedef enum { NSA_F32 = 0, NSA_BF16 = 1 } nsa_dtype;

typedef struct nsa_shape {
  int32_t batch;              /* dense layout: number of sequences (cu_seqlens == NULL)   */
  int32_t seqlen;             /* dense: tokens per sequence; varlen: the longest length   */
  const int32_t* cu_seqlens;  /* device [n_seqs+1], or NULL for the dense layout          */
  int32_t n_seqs;             /* varlen only: number of sequences                        */
  int64_t total_tokens;       /* varlen only: cu_seqlens[n_seqs] (dense: batch*seqlen)   */
  int32_t h, h_kv, d;         /* query heads, kv-heads, head dimension                    */
  nsa_dtype dtype;            /* element type of Q, K, V, O and compressed keys          */
} nsa_shape;

/* Library version string. */
NSA_API const char* nsa_version(void);

/* Message of the last failed call made by this thread ("" if none). */
NSA_API const char* nsa_last_error(void);

/* Device status word of the current device.  Kernels that wait on other warps, copies
 * or CTAs (the tcgen05 branches of nsa_layer_fwd, the TMA-fed selected attention, the
 * decode step's wait for a row's block list) bound every wait to about a second;
 * when one runs out the kernel sets the word to NSA_ERR_TIMEOUT, stops waiting, drains
 * its copies in flight and releases its tensor memory, so the context stays usable; while
 * the word is set, the tcgen05 branches and the decode step skip their work.  Outputs of a
 * call that set the word are not valid.  Runtime error reporting, with no counterpart in
 * the pages.
 *   status  host int32 out: NSA_OK or NSA_ERR_TIMEOUT
 *   reset   nonzero: clear the word after reading it
 * Blocks until the device is idle (a synchronous copy).  Returns NSA_ERR_INVALID for a
 * NULL status, NSA_ERR_CUDA when the copy fails. */
NSA_API nsa_status nsa_device_status(int32_t* status, int reset);

/* Limit of those bounded waits, in nanoseconds, on the current device (0 restores the
 * default of one second).  It applies to the first-level waits (a role waiting for a copy,
 * for the tensor cores or for another CTA's result); the waits with which a kernel that
 * gave up drains its copies and tensor-core work in flight keep the one-second limit.  A
 * diagnostic hook with no counterpart in the pages: a limit far below a wait's normal
 * length makes the waits run out on purpose, so the give-up path (status word, drain,
 * return) can be exercised and the caller's error handling tested.  A limit below one
 * microsecond (finer than the device timer) makes a wait give up at its first
 * unsuccessful probe.
 * Synchronous (a copy to each kernel unit's constant); returns NSA_ERR_CUDA when it fails.
 * Set it only while none of this library's kernels run. */
NSA_API nsa_status nsa_set_wait_limit_ns(uint64_t ns);

/* S1 -- key (or value) compression.  [NOSA-Parts] core component 1: keys are cut into
 * windows of `kernel` tokens at step `stride` and each window is mean-pooled;
 * [NOSA-Triton] "beyond the kernel": kernel 32, stride 16, 50% overlap.
 *   k      [tokens, h_kv, d]            in
 *   k_cmp  [sum_i n_c(L_i), h_kv, d]    out, fp32 mean rounded to nearest (ties even)
 * Windows never cross a sequence boundary.  Requires kernel % stride == 0 and
 * kernel/stride <= 4; h_kv*d a multiple of 8 (bf16) or 4 (fp32). */
NSA_API nsa_status nsa_compress_k(const nsa_shape* shape, const void* k, void* k_cmp, int kernel, int stride,
                          cudaStream_t stream);

/* S2+S3 -- compressed scores pooled to selection blocks.  [NSA-Triton] sec. 1.1 (the
 * selection reuses the compressed-attention scores) and [NOSA-Parts] core component 3,
 * stage 1 (a light attention of q against the compressed keys): for query t, head hh of
 * group g, p[hh,c] = softmax over causal c of scale * q[t,hh].k_cmp[c,g]; the group
 * probability P_g[c] = sum over the group's heads of p[hh,c].  [NOSA-Triton] mechanisms
 * 2-3 (window mean divided by the count of valid entries): the block score of block j is
 * the mean of P_g over the windows inside the block, {c : c*stride >= j*block_size,
 * c*stride + kernel <= (j+1)*block_size}, counting windows c < n_c(L) only (causally
 * masked ones count as zeros); no such window gives 0.
 *   q             [tokens, h, d] bf16
 *   k_cmp         packed compressed keys (nsa_compress_k) bf16
 *   lse_in        nullable [tokens, h] fp32: the natural-log softmax normaliser of each
 *                 (token, head) over its causal compressed keys, as written by
 *                 nsa_cmp_attn_fwd.  Given, the kernel skips its own normaliser pass.
 *   block_scores  [tokens, h_kv, nb_stride] fp32 out; entries j >= n_b(L) are 0.
 * Requires kernel 32, stride 16, block_size 64, d in {64,128}, h/h_kv in {1,2,4,8,16},
 * nb_stride >= n_b(longest sequence). */
NSA_API nsa_status nsa_cmp_scores_pool(const nsa_shape* shape, const void* q, const void* k_cmp, int kernel,
                               int stride, int block_size, float scale, const float* lse_in,
                               float* block_scores, int nb_stride, cudaStream_t stream);

/* S4 -- top-k block selection.  [NOSA-Triton] "beyond the kernel": keep the
 * n_init initial blocks and the n_local local blocks (ending at the query's own block
 * t / block_size) as forced candidates, exclude blocks that start after t, take the k
 * best by score and return them sorted.  Forced blocks rank above every score; equal
 * scores rank the lower block index first; k counts the forced blocks; when fewer than k
 * blocks are causal the list is padded with -1 at the end.
 *   block_scores   [tokens, h_kv, nb_stride] fp32 (finite) in
 *   block_indices  [tokens, h_kv, k] int32 out, ascending, -1 padded
 * Requires 1 <= k <= 64 and nb_stride <= 2048. */
NSA_API nsa_status nsa_topk_select(const nsa_shape* shape, const float* block_scores, int nb_stride,
                           int block_size, int n_init, int n_local, int k, int32_t* block_indices,
                           cudaStream_t stream);

/* S2-S4 in one call -- block selection from the compressed keys: the block scores of
 * nsa_cmp_scores_pool (kept in the workspace, never returned) followed by
 * nsa_topk_select, with the same definitions, arguments and limits ([NOSA-Parts] core
 * component 3, first stage; [NOSA-Triton] beyond the kernel).
 *   q              [tokens, h, d]; k_cmp [sum_i n_c(L_i), h_kv, d]
 *   block_indices  [tokens, h_kv, k] int32 out, ascending, -1 padded
 *   workspace      device, >= nsa_select_workspace_size(shape, block_size) bytes,
 *                  256-byte aligned, caller-owned; its contents are scratch
 * Requires kernel 32, stride 16, block_size 64, bf16, d in {64, 128}, h/h_kv in
 * {1, 2, 4, 8, 16}, 1 <= k <= 64, sequences up to 131072 tokens. */
NSA_API size_t nsa_select_workspace_size(const nsa_shape* shape, int block_size);
NSA_API nsa_status nsa_select(const nsa_shape* shape, const void* q, const void* k_cmp, int kernel, int stride,
                              int block_size, float scale, int n_init, int n_local, int k,
                              int32_t* block_indices, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream);

/* S5 -- selected-block attention (prefill).  [TileLang-NSA] sec. 2: for each entry of
 * the query's list the block starting at i_s = index * block_size is used when
 * 0 <= i_s <= t; keys past t inside it are masked; every query head of a GQA group reads
 * the same block list ([NSA-Triton] sec. 1.2, group-centric loading).  Softmax in fp32
 * with base-2 exponentials of scale*log2(e)-folded scores ([TileLang-NSA] sec. 3.1).
 *   q, o           [tokens, h, d]; k, v [tokens, h_kv, d]
 *   block_indices  [tokens, h_kv, S] int32; -1 and non-causal entries are skipped; an
 *                  index listed twice is attended twice
 *   lse            nullable [tokens, h] fp32 out: natural-log softmax normaliser (-inf
 *                  and o = 0 when no key is selected)
 * bf16: d in {64,128}, block_size in {16,32,64}, S <= 64, h/h_kv <= 16 or a multiple
 * of 16.  fp32: d <= 256, S*block_size <= 4096. */
NSA_API nsa_status nsa_sparse_fwd(const nsa_shape* shape, const void* q, const void* k, const void* v,
                          const int32_t* block_indices, int S, int block_size, float scale, void* o,
                          float* lse, cudaStream_t stream);

/* Backward of S7, the compressed branch: gradients for an upstream dO of the attention
 * over the stored compressed keys and values (the forward nsa_cmp_attn_fwd).  Per (token,
 * head) row over its causal compressed keys c < n_causal(t): p_c = exp(scale q.kc_c -
 * lse), dp_c = dO.vc_c, D = dO.o, ds_c = p_c (dp_c - D); dq = scale sum ds_c kc_c,
 * dk_cmp[c] += scale ds_c q, dv_cmp[c] += p_c dO.  Rows without causal keys give dq = 0.
 * The pages print the forward only ([NSA-Triton] sec. 1.1); this is its derivative.
 *   q, o, d_o, dq    [tokens, h, d] bf16;  lse [tokens, h] fp32 (the forward's)
 *   k_cmp, v_cmp, dk_cmp, dv_cmp  [n_cmp_total, h_kv, d] bf16, packed per sequence
 *   workspace        nsa_cmp_attn_bwd_workspace_size() bytes, 256-byte aligned
 * Deterministic.  Requires bf16, d 128, h/h_kv <= 16, at most 4096 compressed keys per
 * sequence. */
NSA_API size_t nsa_cmp_attn_bwd_workspace_size(const nsa_shape* shape, int kernel, int stride);
NSA_API nsa_status nsa_cmp_attn_bwd(const nsa_shape* shape, const void* q, const void* k_cmp, const void* v_cmp,
                                    int kernel, int stride, float scale, const void* o, const float* lse,
                                    const void* d_o, void* dq, void* dk_cmp, void* dv_cmp, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream);

/* Backward of S8, the sliding window: the derivative of nsa_swa_fwd for an upstream dO
 * (keys max(0, t-window+1) .. t; the formulas of nsa_sparse_bwd).  Arguments and layouts
 * as nsa_sparse_bwd without the lists; workspace nsa_swa_bwd_workspace_size() bytes.
 * Requires bf16, d 128, h/h_kv <= 16, 1 <= window <= 1984. */
NSA_API size_t nsa_swa_bwd_workspace_size(const nsa_shape* shape, int window);
NSA_API nsa_status nsa_swa_bwd(const nsa_shape* shape, const void* q, const void* k, const void* v, int window,
                               float scale, const void* o, const float* lse, const void* d_o, void* dq, void* dk,
                               void* dv, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Backward of S9, the gate combine: with g_i = sigmoid(a_i) and o = sum_i g_i o_i, the
 * branch gradients are g_i dO and the logit gradients g_i (1 - g_i) (dO . o_i).
 *   d_o, o_cmp, o_slc, o_swa, d_cmp, d_slc, d_swa  [tokens, h, d] bf16
 *   gate_logits, d_gate_logits  [tokens, h, 3] fp32.  d % 8 == 0, d <= 256. */
NSA_API nsa_status nsa_gate_combine_bwd(int64_t tokens, int h, int d, const void* d_o, const void* o_cmp,
                                        const void* o_slc, const void* o_swa, const float* gate_logits, void* d_cmp,
                                        void* d_slc, void* d_swa, float* d_gate_logits, cudaStream_t stream);

/* Backward of S1, the mean pooling: token row t of a sequence receives, from every
 * compressed window c of that sequence containing it (c*stride <= t < c*stride+kernel),
 * the window's gradient divided by kernel; tokens in no window get 0.
 *   dk_cmp [n_cmp_total, h_kv, d] bf16;  dk [tokens, h_kv, d] bf16 out.  d % 8 == 0. */
NSA_API nsa_status nsa_compress_bwd(const nsa_shape* shape, const void* dk_cmp, int kernel, int stride, void* dk,
                                    cudaStream_t stream);

/* NOSA stage 2 -- pooled importance scores per block.  [NOSA-Parts] core component 2:
 * a scorer gives every key position an importance score (CIS; produced elsewhere, e.g.
 * by a learned scorer); [NOSA-Triton] mechanisms 1-3: the scores are mean-pooled over
 * windows of `kernel` positions at step `stride`, aligned with the key compressor (full
 * windows, n_c(L) of them); [NOSA-Parts] core component 3: the window means are brought
 * to blocks with the rule of S3 (block j averages the windows lying inside it; no
 * window -> 0).
 *   cis  [tokens, h_kv] fp32;  out [n_seqs, h_kv, nb_stride] fp32, 0 past n_b(L). */
NSA_API nsa_status nsa_cis_block_scores(const nsa_shape* shape, const float* cis, int kernel, int stride,
                                        int block_size, int nb_stride, float* out, cudaStream_t stream);

/* NOSA two-stage selection ([NOSA-Parts] core component 3).  Stage 1: the forced blocks
 * and the best blocks by attention block score, qk_select in all (nsa_topk_select with
 * k = qk_select).  Stage 2: those blocks ranked by their block CIS score (forced blocks
 * first, equal scores to the lower block index); the best k are returned ascending,
 * -1 padded.
 *   block_scores      [tokens, h_kv, nb_stride] fp32 (nsa_cmp_scores_pool)
 *   cis_block_scores  [n_seqs, h_kv, nb_stride] fp32 (nsa_cis_block_scores)
 *   block_indices     [tokens, h_kv, k] int32 out
 * Requires 1 <= k <= qk_select <= 64, nb_stride <= 2048. */
NSA_API nsa_status nsa_topk_two_stage(const nsa_shape* shape, const float* block_scores, int nb_stride,
                                      const float* cis_block_scores, int block_size, int n_init, int n_local,
                                      int qk_select, int k, int32_t* block_indices, cudaStream_t stream);

/* NOSA sparse_forward -- selected attention with CIS-scaled values and the all-ones
 * normaliser ([NOSA-Parts] "decoding over only 64 KV blocks": scaled_v = v * cis, and the
 * output divided by the same attention of all-ones values scaled alike).  With p the
 * softmax over the listed keys and c_e the CIS of key e (per kv-head):
 * o = sum_e p_e c_e v_e / sum_e p_e c_e;  lse = log sum_e exp(s_e) c_e.  A row whose
 * weights sum to 0 gets o = 0, lse = -inf.  Lists as in nsa_sparse_fwd.
 *   cis [tokens, h_kv] fp32 (>= 0);  other arguments as nsa_sparse_fwd.
 * Requires bf16, d in {64,128}, block_size 64, S <= 64, h/h_kv <= 16 or a multiple of 16. */
NSA_API nsa_status nsa_sparse_cis_fwd(const nsa_shape* shape, const void* q, const void* k, const void* v,
                                      const float* cis, const int32_t* block_indices, int S, int block_size,
                                      float scale, void* o, float* lse, cudaStream_t stream);

/* Backward of S5: gradients of the selected-block attention for an upstream gradient
 * dO.  The pages train with the selected branch ([NSA-Triton] sec. 4) and print its
 * forward only ([TileLang-NSA] sec. 2); this is the derivative of that forward.  Per
 * (token, head) row with list keys e (as in nsa_sparse_fwd, an index listed twice
 * counts twice): p_e = exp(scale q.k_e - lse), dp_e = dO.v_e, D = dO.o,
 * ds_e = p_e (dp_e - D); dq = scale sum_e ds_e k_e, dk[e] += scale ds_e q,
 * dv[e] += p_e dO.
 *   q, o, d_o, dq  [tokens, h, d] bf16;  k, v, dk, dv  [tokens, h_kv, d] bf16
 *   block_indices  [tokens, h_kv, S] int32 (the forward's lists)
 *   o, lse         the forward's outputs for the same inputs (lse [tokens, h] fp32)
 *   workspace      device scratch of nsa_sparse_bwd_workspace_size() bytes, 256-byte
 *                  aligned, owned by the caller (fp32 partial sums of dk and dv per
 *                  (sequence, kv-head, key block, 2048-query chunk), and D)
 * dk and dv are written for every key row (0 where no query selects it).  Results are
 * deterministic (fixed summation order; no floating-point atomics).
 * Requires bf16, d 128, block_size 64, S <= 64, h/h_kv <= 16. */
NSA_API size_t nsa_sparse_bwd_workspace_size(const nsa_shape* shape, int S, int block_size);
NSA_API nsa_status nsa_sparse_bwd(const nsa_shape* shape, const void* q, const void* k, const void* v,
                                  const int32_t* block_indices, int S, int block_size, float scale, const void* o,
                                  const float* lse, const void* d_o, void* dq, void* dk, void* dv, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/* Block-mask sparse attention (the block-sparse companion of the pages' native sparse
 * attention).  [TileLang-NSA] sec. 1, block-sparse attention: the attention matrix is
 * cut into block_size x block_size tiles and a mask marks the active ones; only active
 * tiles are computed; is_causal keeps the lower triangle.  Query (b, t, head h) attends
 * every key of every key block kb with block_mask[b, h, t / block_size, kb] != 0
 * (restricted to keys <= t when causal); a query without any attended key gets o = 0,
 * lse = -inf.
 *   q, k, v, o  [batch, seqlen, h, d]: dense layout (cu_seqlens NULL), multi-head K/V
 *               (h_kv == h)
 *   block_mask  uint8 [batch, h, n, n], n = seqlen / block_size, device
 *   lse         nullable [batch * seqlen, h] fp32 out (natural log)
 *   workspace   >= nsa_block_sparse_workspace_size(shape) bytes, 256-byte aligned:
 *               V transposed per head for the tensor-core PV operand
 * Requires bf16, d = 128, block_size = 64, seqlen a multiple of 64 and <= 65536. */
NSA_API size_t nsa_block_sparse_workspace_size(const nsa_shape* shape);
NSA_API nsa_status nsa_block_sparse_fwd(const nsa_shape* shape, const void* q, const void* k, const void* v,
                                        const uint8_t* block_mask, int block_size, int causal, float scale,
                                        void* o, float* lse, void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream);

/* S7 -- compressed-attention branch.  [NSA-Triton] sec. 1.1 and 2.2 (taken as the
 * definition): softmax over the causal compressed keys of scale * q.k_cmp, weighted sum
 * of v_cmp.  A query with no causal compressed key gets o = 0 and lse = -inf.
 *   k_cmp, v_cmp   packed compressed keys / values (nsa_compress_k on K and on V), exactly
 *                  the packed rows of the sequences (tiles reaching past them are read with
 *                  bounds checks)
 *   o [tokens, h, d] out; lse nullable [tokens, h] fp32 out (natural log)
 *   workspace      nsa_cmp_attn_fwd_workspace_size() bytes, 256-byte aligned (V transposed
 *                  for the tensor cores); NULL allowed when that size is 0
 * bf16 only; d in {64,128}; h/h_kv divides 16 or is a multiple of 16.  d = 128 with h/h_kv a
 * power of two runs on the tcgen05 tensor cores (the layer's kernel); other shapes on
 * mma.sync, with no workspace. */
NSA_API size_t nsa_cmp_attn_fwd_workspace_size(const nsa_shape* shape, int kernel, int stride);
NSA_API nsa_status nsa_cmp_attn_fwd(const nsa_shape* shape, const void* q, const void* k_cmp,
                            const void* v_cmp, int kernel, int stride, float scale, void* o, float* lse,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* S8 -- sliding-window branch ([NSA-Triton] sec. 1.1: the most recent tokens): keys
 * max(0, t-window+1) .. t.  Same layouts, limits and kernel choice as nsa_cmp_attn_fwd;
 * workspace of nsa_swa_fwd_workspace_size() bytes. */
NSA_API size_t nsa_swa_fwd_workspace_size(const nsa_shape* shape);
NSA_API nsa_status nsa_swa_fwd(const nsa_shape* shape, const void* q, const void* k, const void* v,
                       int window, float scale, void* o, float* lse, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* S9 -- gate combine ([NSA-Triton] sec. 1.1: gates[0]*compressed + gates[1]*selected +
 * gates[2]*local), each gate the logistic sigmoid of its logit.
 *   o_cmp, o_slc, o_swa, o  [tokens, h, d] bf16;  gate_logits [tokens, h, 3] fp32.
 * o may alias any input.  d a multiple of 8. */
NSA_API nsa_status nsa_gate_combine(int64_t tokens, int h, int d, const void* o_cmp, const void* o_slc,
                            const void* o_swa, const float* gate_logits, void* o,
                            cudaStream_t stream);

/* S6 -- one decode step.  [NOSA-Parts] "how decoding uses only 64 KV blocks": the
 * newest query of each sequence (position L_b - 1; the cache already holds its key and
 * value) is scored against the compressed keys (S2, S3), k blocks are chosen (S4) and
 * attention runs over the chosen blocks only (S5).
 *   seqlens      device int32 [batch], 1 <= L_b <= max_len
 *   q, o         [batch, h, d] bf16
 *   k_cache, v_cache  [batch, max_len, h_kv, d] bf16, in device memory or in page-locked
 *                host memory ([NOSA-Parts] "core idea": the KV cache is offloaded to host
 *                memory and only the chosen blocks come back).  A host cache must come from
 *                cudaHostAlloc or cudaHostRegister; the chosen blocks are then read over the
 *                CPU-GPU link straight into shared memory, with no device copy of the cache.
 *                Pageable host memory is rejected with NSA_ERR_INVALID.
 *   k_cmp_cache  [batch, n_c(max_len), h_kv, d] bf16; rows c < n_c(L_b) valid; device or
 *                page-locked host memory (keep it on the device: every step reads all of it)
 *   idx_out      nullable [batch, h_kv, k] int32: the chosen blocks
 *   workspace    device scratch of nsa_sparse_decode_workspace_size() bytes, 256-byte
 *                aligned, owned by the caller, not read before it is written
 * Requires kernel 32, stride 16, block_size 64, d 128, h/h_kv in {1,2,4,8,16}, k <= 64,
 * max_len <= 65536. */
NSA_API size_t nsa_sparse_decode_workspace_size(int batch, int max_len, int h, int h_kv, int d, int kernel,
                                        int stride, int block_size, int k);
NSA_API nsa_status nsa_sparse_decode(int batch, const int32_t* seqlens, int max_len, int h, int h_kv, int d,
                             const void* q, const void* k_cache, const void* v_cache,
                             const void* k_cmp_cache, int kernel, int stride, int block_size,
                             int n_init, int n_local, int k, float scale, int32_t* idx_out, void* o,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* The NOSA decode step ([NOSA-Parts] "decoding over only 64 KV blocks", core component
 * 3): nsa_sparse_decode with the CIS-weighted attention of nsa_sparse_cis_fwd over the
 * chosen blocks, and, when cis_block_scores is given, the two-stage selection of
 * nsa_topk_two_stage (stage 1 keeps the forced blocks and the best qk_select blocks by
 * attention score, stage 2 keeps the k best of those by block CIS score).
 *   cis_cache         [batch, max_len, h_kv] fp32 (>= 0), device or page-locked host memory
 *   cis_block_scores  nullable [batch, h_kv, nb_stride] fp32: the block CIS scores of each
 *                     sequence (nsa_cis_block_scores over the sequence's own length; only
 *                     the blocks that stage 1 can keep are read: with n_local >= 1 the
 *                     query's own block is forced, and a dense call over the padded cache
 *                     gives the same selection)
 * Other arguments, workspace (nsa_sparse_decode_workspace_size) and limits as
 * nsa_sparse_decode; k <= qk_select <= 64 when cis_block_scores is given. */
NSA_API nsa_status nsa_sparse_decode_cis(int batch, const int32_t* seqlens, int max_len, int h, int h_kv, int d,
                                         const void* q, const void* k_cache, const void* v_cache,
                                         const void* k_cmp_cache, const float* cis_cache,
                                         const float* cis_block_scores, int nb_stride, int qk_select, int kernel,
                                         int stride, int block_size, int n_init, int n_local, int k, float scale,
                                         int32_t* idx_out, void* o, void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream);

/* Allocation-free variant of nsa_sparse_decode, for callers that cannot allocate device
 * memory when they run a decode step (code inside an allocator or memory-pool callback,
 * runtimes that pre-reserve all device memory, plug-ins handed only their input and
 * output buffers).  The pages have no counterpart: this is an interface convenience.
 * Same arguments, kernels and results as nsa_sparse_decode, without the workspace: the
 * scratch is a fixed array of nsa_sparse_decode_noalloc_max_bytes() bytes (16 MiB) in
 * device memory that the library owns; every GPU that loads the library holds it until
 * the process exits.  The caller still passes inputs and outputs.
 *   - Sizes the decode step does not support are rejected first, with the status and
 *     message of nsa_sparse_decode.  Supported steps whose
 *     nsa_sparse_decode_workspace_size() exceeds the fixed size are then rejected with
 *     NSA_ERR_UNSUPPORTED and a message naming both sizes.
 *   - The first call on a device looks up the array's device address (a CUDA runtime
 *     symbol query, no allocation); make that first call before any stream capture.  The
 *     address is kept per device and CUDA context: after a device reset (a new context,
 *     with a new copy of the array) the next call looks it up again.
 *   - All calls share the one array, which keeps the last call's contents; every byte a
 *     call reads is written earlier in the same call, so nothing needs clearing.  Calls
 *     that overlap on the GPU (other streams, other host threads) race on it: order them.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine. */
NSA_API size_t nsa_sparse_decode_noalloc_max_bytes(void);
NSA_API nsa_status nsa_sparse_decode_noalloc(int batch, const int32_t* seqlens, int max_len, int h, int h_kv,
                                             int d, const void* q, const void* k_cache, const void* v_cache,
                                             const void* k_cmp_cache, int kernel, int stride, int block_size,
                                             int n_init, int n_local, int k, float scale, int32_t* idx_out,
                                             void* o, cudaStream_t stream);

/* Full three-branch layer forward ([NSA-Triton] sec. 1.1): compress K and V (S1), the
 * compressed branch (S7, which also yields the normaliser reused by the selection),
 * block scores from the same compressed probabilities (S2, S3), top-S selection (S4),
 * the selected branch (S5), the sliding-window branch (S8) and the gated sum (S9).
 *   q, o [tokens, h, d] bf16; k, v [tokens, h_kv, d] bf16; gate_logits [tokens, h, 3]
 *   idx_out nullable [tokens, h_kv, S] int32 (the chosen blocks)
 *   workspace of nsa_layer_fwd_workspace_size() bytes (256-byte aligned)
 * Limits: those of the calls above. */
NSA_API size_t nsa_layer_fwd_workspace_size(const nsa_shape* shape, int kernel, int stride, int block_size,
                                    int S);
NSA_API nsa_status nsa_layer_fwd(const nsa_shape* shape, const void* q, const void* k, const void* v,
                         const float* gate_logits, int kernel, int stride, int block_size, int S,
                         int n_init, int n_local, int window, float scale, void* o, int32_t* idx_out,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Training pair for the full layer.  nsa_layer_fwd_train is nsa_layer_fwd (same
 * arguments, limits, workspace and output) that also keeps, in the caller's buffers, what
 * the backward needs; nsa_layer_bwd then returns the gradients of the layer output o with
 * respect to q, k, v and the gate logits for an upstream d_o.  The backward chains the
 * gate backward, the backward of each branch (nsa_cmp_attn_bwd with nsa_compress_bwd for
 * the pooling of both K and V, nsa_sparse_bwd on the kept block lists, which the
 * selection does not differentiate through, and nsa_swa_bwd) and sums dq, dk, dv over the
 * branches.  The pages train with this layer ([NSA-Triton] sec. 4) and print its forward
 * only; the backward is the forward's derivative.
 * Buffers of nsa_layer_saved (all device memory, owned by the caller, written by the
 * training forward, read by the backward):
 *   k_cmp, v_cmp  [n_cmp_total, h_kv, d] bf16 (n_cmp_total = sum of n_c(L) per sequence)
 *   o_cmp, o_slc, o_swa  [tokens, h, d] bf16 (branch outputs before the gate)
 *   lse_cmp, lse_slc, lse_swa  [tokens, h] fp32;  idx [tokens, h_kv, S] int32
 * nsa_layer_bwd: d_o, dq [tokens, h, d]; dk, dv [tokens, h_kv, d] (bf16);
 * d_gate_logits [tokens, h, 3] fp32; workspace of nsa_layer_bwd_workspace_size() bytes,
 * 256-byte aligned.  Requires d 128, window <= 1984, at most 4096 compressed keys per
 * sequence, plus the limits of nsa_layer_fwd. */
typedef struct nsa_layer_saved {
  void* k_cmp;
  void* v_cmp;
  void* o_cmp;
  void* o_slc;
  void* o_swa;
  float* lse_cmp;
  float* lse_slc;
  float* lse_swa;
  int32_t* idx;
} nsa_layer_saved;

NSA_API nsa_status nsa_layer_fwd_train(const nsa_shape* shape, const void* q, const void* k, const void* v,
                                       const float* gate_logits, int kernel, int stride, int block_size, int S,
                                       int n_init, int n_local, int window, float scale, void* o,
                                       const nsa_layer_saved* saved, void* workspace, size_t workspace_bytes,
                                       cudaStream_t stream);
NSA_API size_t nsa_layer_bwd_workspace_size(const nsa_shape* shape, int kernel, int stride, int block_size, int S,
                                            int window);
NSA_API nsa_status nsa_layer_bwd(const nsa_shape* shape, const void* q, const void* k, const void* v,
                                 const float* gate_logits, int kernel, int stride, int block_size, int S, int window,
                                 float scale, const nsa_layer_saved* saved, const void* d_o, void* dq, void* dk,
                                 void* dv, float* d_gate_logits, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NSA_H_ */
