/*
 * fa.h — C ABI of libfa.so: exact IO-aware softmax attention on GB300 (sm_103a).
 *
 * What is computed.  For every batch b and head h, with scale σ (normally 1/√d):
 *     S = σ·Q Kᵀ,  P = softmax(S) row-wise,  O = P V,  LSE_i = m_i + ln ℓ_i
 * where m_i is the row max of S and ℓ_i = Σ_j e^(S_ij − m_i).  This is the
 * standard attention of "FlashAttention：IO-aware 的注意力 kernel"
 * (inference-learning-path.pages.dev) §3.1, computed the way its §3.2 describes:
 * key/value tiles stream through on-chip memory while each query row keeps a
 * running max m, running normaliser ℓ and an unnormalised accumulator, all
 * rescaled by e^(m_old − m_new) when the max moves; O/ℓ is taken once at the
 * end, so the N×N score and probability matrices never reach device memory.
 *
 * Conventions shared by every entry point.
 *   - Tensors are device pointers (fa_forward_host alone takes host ones).  Q, K, V, O, dO, dQ, dK, dV are
 *     [B, H, N, d] row-major with d innermost, the shape "Q, K, V ∈ R^{N×d}"
 *     of the FlashAttention walkthrough (kyonqi.github.io, "Flash Attention
 *     Forward") with batch and head dims in front.  LSE is [B, H, N] float32.
 *   - LSE uses the natural log of the scaled scores.
 *   - fa_dtype selects the storage type of Q, K, V, O (and dO, dQ, dK, dV).
 *     FA_BF16 tensors accumulate in fp32; FA_FP32 computes in fp32 throughout.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call is asynchronous on that stream; a call returns after its
 *     kernels are enqueued.
 *   - The caller owns and allocates every buffer, including workspaces whose
 *     size is queried first.  The library allocates no device memory.
 *   - Errors.  FA_ERR_INVALID_ARG: null pointer, non-positive size, bad
 *     stride, misaligned pointer (16-byte alignment is required), scale not
 *     finite and > 0, workspace too small.  FA_ERR_UNSUPPORTED: a head dim,
 *     dtype or size the library has no kernel for; there is never a silent
 *     fallback to another algorithm.  FA_ERR_CUDA: a launch or earlier
 *     asynchronous CUDA error.  FA_ERR_DEVICE_TIMEOUT: a kernel gave up on a
 *     pipeline wait (reported by fa_device_status).  On any error the
 *     message is available from fa_get_last_error() in the calling thread.
 *     Validation happens before anything is enqueued, so an argument error
 *     leaves the stream untouched.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,
  FA_ERR_UNSUPPORTED = 2,
  FA_ERR_CUDA = 3,
  FA_ERR_DEVICE_TIMEOUT = 4
} fa_status;

typedef enum fa_dtype { FA_BF16 = 0, FA_FP32 = 1 } fa_dtype;

/* Attention mask.  FA_MASK_CAUSAL is the causal mask the lesson's memory lab
 * uses (§5, is_causal=True), aligned to the bottom-right corner: query row i of
 * N_q sees keys j <= i + (N_kv − N_q); it needs N_q <= N_kv so no row is empty. */
typedef enum fa_mask { FA_MASK_NONE = 0, FA_MASK_CAUSAL = 1 } fa_mask;

/* Version of this ABI; bumped on any incompatible change. */
FA_API int fa_abi_version(void);

/*
 * fa_forward — tiled forward pass, one write of O and LSE.
 *   Follows the lesson's §2 mental model and §3.2 recurrence; the statistics it
 *   saves are the ones the walkthrough's "Flash Attention Backward" section
 *   keeps for the backward (here folded into LSE = m + ln ℓ).
 *   q [B,H,N_q,d], k and v [B,H,N_kv,d]; o [B,H,N_q,d] (same dtype as q);
 *   lse [B,H,N_q] float32 (may be NULL to skip it).
 *   strides: NULL for contiguous tensors, or 12 element strides
 *   {q_b, q_h, q_n, k_b, k_h, k_n, v_b, v_h, v_n, o_b, o_h, o_n}; the d stride is
 *   always 1 and every stride × element size must be a multiple of 16 bytes.
 *   N_q may differ from N_kv (query rows are independent).  No mask.
 *   Supported: FA_BF16 with d ∈ {64, 128} (tensor-core kernel) and FA_FP32 with
 *   d ∈ {64, 128} (fp32 CUDA-core kernel, for exact checks).
 */
FA_API fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int N_q, int N_kv, int d, fa_dtype dtype, float scale,
                     const int64_t* strides, void* stream);

/*
 * fa_forward_masked — fa_forward with a mask (FA_MASK_NONE is fa_forward).
 *   With FA_MASK_CAUSAL masked scores are −∞ before the softmax; a CTA streams
 *   only the key tiles its rows can see.  N_q > N_kv with a causal mask gives
 *   FA_ERR_INVALID_ARG; a causal N_q above 65535·256 gives FA_ERR_UNSUPPORTED.
 *   Same arguments, layouts and support as fa_forward.
 */
FA_API fa_status fa_forward_masked(const void* q, const void* k, const void* v, void* o, float* lse,
                                   int B, int H, int N_q, int N_kv, int d, fa_dtype dtype, float scale,
                                   const int64_t* strides, fa_mask mask, void* stream);

/*
 * fa_forward_fp8 — forward with FP8 (E4M3) inputs, FlashAttention-3's addition
 *   (lesson §3.3; interview notes §四.5).  q, k, v hold E4M3 codes (one byte
 *   each, [B,H,N,d] contiguous) whose true values are q_descale·q, k_descale·k,
 *   v_descale·v; the MMAs run as tcgen05 kind::f8f6f4 with fp32 accumulation,
 *   P̃ is rounded to E4M3 for the P̃V product while ℓ sums the unrounded fp32
 *   values, and o is written as bf16 [B,H,N_q,d] with lse fp32 as in fa_forward.
 *   mask: FA_MASK_NONE or FA_MASK_CAUSAL.  Supported: d = 128.
 */
FA_API fa_status fa_forward_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int N_q, int N_kv, int d, float scale, float q_descale,
                                float k_descale, float v_descale, fa_mask mask, void* stream);

/*
 * fa_forward_host_workspace_size — device bytes fa_forward_host needs for the
 *   same arguments: two chunk buffers, each holding q [heads,N_q,d], k and v
 *   [heads,N_kv,d], o [heads,N_q,d] (element size of dtype) and lse [heads,N_q]
 *   float32 for `heads` = min(heads_per_chunk, B·H) (heads_per_chunk = 0: the
 *   chunk fa_forward_host picks on the current device), every piece rounded up
 *   to 256 bytes.  Returns 0 for invalid sizes or dtype, or when
 *   heads_per_chunk = 0 and no device can be queried.
 */
FA_API size_t fa_forward_host_workspace_size(int B, int H, int N_q, int N_kv, int d, fa_dtype dtype,
                                             int heads_per_chunk);

/*
 * fa_forward_host — fa_forward_masked on HOST tensors.  The lesson states the
 *   forward on HBM-resident Q, K, V (§1–§3); this entry point adds the transfer
 *   to and from host memory, which it does not cover.  q, k, v, o,
 *   lse are host pointers to contiguous [B,H,N,d] tensors (lse [B,H,N_q]
 *   float32, may be NULL), preferably page-locked: copies from pageable memory
 *   are correct but do not overlap.  The B·H heads are processed in chunks of
 *   heads_per_chunk (0 = let the library choose) through two device buffers in
 *   `workspace` (>= fa_forward_host_workspace_size bytes, 256-byte aligned,
 *   owned by the caller): the copy of chunk c+1 in, the forward on chunk c and
 *   the copy of chunk c−1 out run concurrently on two library-owned copy
 *   streams and `stream`, ordered after the work already queued on `stream`.
 *   The call returns once everything is queued; o and lse are valid after
 *   `stream` has been synchronised.  Results equal fa_forward_masked's on the
 *   same data.  Calls on one device are serialised internally: outside graph
 *   capture, a call's first copy in waits until the previous call has copied
 *   its results out, so eager calls from several threads or streams may share
 *   one workspace.  A captured call is not ordered against other calls: its
 *   replays need a workspace of their own, or ordering by the caller.  Argument errors
 *   return FA_ERR_INVALID_ARG before anything is queued; dtype, d and mask as
 *   for fa_forward_masked.
 */
FA_API fa_status fa_forward_host(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H, int N_q, int N_kv, int d, fa_dtype dtype, float scale,
                                 fa_mask mask, int heads_per_chunk, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * fa_decode_choose_splits — a split count for the decode entry points that keeps
 *   the GPU busy without making chunks too short: about 27 CTAs per SM for
 *   single-head decode (three are resident per SM), about one per SM for
 *   grouped decode (H_q > H_kv, one resident per SM), at least 256 keys per
 *   split, rounded to a power of two and clamped to [1, 256].  Fitted to
 *   measurements on GB300; uses the current device's SM count (152 if none can
 *   be queried).  Returns 0 for non-positive sizes or H_q not a multiple of H_kv.
 */
FA_API int fa_decode_choose_splits(int B, int H_q, int H_kv, int N_kv);

/*
 * fa_decode_workspace_size — bytes of workspace fa_decode_splitkv needs:
 *   the partial outputs B·H·n_splits·d·4 bytes and the partial (m, ℓ) pairs
 *   B·H·n_splits·2·4 bytes, each rounded up to a multiple of 256.
 */
FA_API size_t fa_decode_workspace_size(int B, int H, int d, int n_splits);

/*
 * fa_decode_splitkv — one query row per head (S_q = 1) against N_kv keys.
 *   The key range is cut into n_splits contiguous chunks of ceil(N_kv/n_splits)
 *   keys, processed in parallel ("FlashDecoding", lesson §3.3 and §9: split
 *   along the KV length to fill the SMs).  Each chunk c yields an unnormalised
 *   triple (m_c, ℓ_c, o_c); a second kernel folds the triples with the
 *   block-merge rule of the FlashAttention interview notes (omica.com.cn
 *   news 1422242, §二.3):  m = max(m_a, m_b), ℓ = ℓ_a e^(m_a−m) + ℓ_b e^(m_b−m),
 *   o = o_a e^(m_a−m) + o_b e^(m_b−m), and writes O = o/ℓ and LSE = m + ln ℓ.
 *   q [B,H,1,d], k and v [B,H,N_kv,d] contiguous; o [B,H,1,d]; lse [B,H] (or NULL).
 *   workspace: device buffer of at least fa_decode_workspace_size() bytes, used
 *   for the partial triples; its contents on entry do not matter.
 *   Supported: FA_BF16, d = 64 or 128, 1 ≤ n_splits ≤ 256.
 */
FA_API fa_status fa_decode_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int N_kv, int d, fa_dtype dtype, float scale,
                            int n_splits, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_decode_splitkv_gqa — fa_decode_splitkv with grouped query heads.
 *   H_q query heads share H_kv key/value heads: query head h reads key/value
 *   head h / (H_q / H_kv), the grouped-query layout of the model whose shapes
 *   the lesson's lab uses (Qwen2.5-7B: 28 query heads, 4 key/value heads).  One
 *   CTA per (b, key/value head, chunk) reads each K/V byte once for the whole
 *   group: with G = 1 this is fa_decode_splitkv; with G >= 2 the group's query
 *   rows go through tcgen05 MMAs (S = Q_g K_jᵀ, O += P̃ V_j), because 2·G·d
 *   multiply-adds per key would outrun CUDA cores long before the HBM stream.
 *   q [B,H_q,1,d], k and v [B,H_kv,N_kv,d] contiguous; o [B,H_q,1,d]; lse [B,H_q]
 *   (or NULL).  workspace: fa_decode_workspace_size(B, H_q, d, n_splits) bytes.
 *   Supported: FA_BF16, d = 64 or 128, H_q = G·H_kv with 1 <= G <= 128 (G = H_q is
 *   multi-query attention), 1 ≤ n_splits ≤ 256.
 */
FA_API fa_status fa_decode_splitkv_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                                       int B, int H_q, int H_kv, int N_kv, int d, fa_dtype dtype, float scale,
                                       int n_splits, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_decode_paged — split-KV decode over a paged key/value cache.
 *   The lesson's vLLM read-along (§4) notes that the fused kernel receives the
 *   paged K/V cache together with its block tables.  Layout chosen here: each
 *   page holds block_size consecutive keys of one key/value head,
 *     k_cache, v_cache  [num_blocks, H_kv, block_size, d]  bf16
 *     block_table       [B, max_blocks] int32: page ids of sequence b, in order
 *     seq_lens          [B] int32: keys of sequence b (1 ≤ len ≤ max_blocks·block_size)
 *   so logical key t of sequence b is row t % block_size of page
 *   block_table[b][t / block_size].  Each sequence's keys are cut into n_splits
 *   chunks of a multiple of 128 keys; partials are merged as in
 *   fa_decode_splitkv.  Query heads may be grouped as in fa_decode_splitkv_gqa.
 *   Page ids outside [0, num_blocks) and lengths outside the table are caught on
 *   the device: page 0 is read instead, and fa_device_status then reports
 *   FA_ERR_INVALID_ARG.  Cache slots past a sequence's end may hold anything.
 *   q [B,H_q,1,d]; o [B,H_q,1,d]; lse [B,H_q] (or NULL); workspace as for
 *   fa_decode_splitkv with H = H_q.
 *   Supported: FA_BF16, d = 64 or 128, block_size ∈ {16, 32, 64, 128}, H_q = G·H_kv, G ≤ 128,
 *   num_blocks·H_kv ≤ 2^31 − 1 (FA_ERR_UNSUPPORTED otherwise).
 */
FA_API fa_status fa_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                                 const int32_t* seq_lens, void* o, float* lse, int B, int H_q, int H_kv,
                                 int num_blocks, int block_size, int max_blocks, int d, fa_dtype dtype, float scale,
                                 int n_splits, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_decode_splitkv_noalloc — fa_decode_splitkv for callers that cannot pass a
 * workspace.  The pages have no counterpart: this is a deployment variant.
 *   Who it is for: callers that cannot allocate device memory when they decode,
 *   e.g. a serving process whose KV cache has reserved nearly all of the GPU's
 *   memory up front (a cudaMalloc at decode time would fail or force a
 *   synchronising reallocation), or a host program that reaches the library
 *   only through this C function and has no device allocator of its own.
 *   Arguments and results are those of fa_decode_splitkv without `workspace`
 *   and `workspace_bytes`.  The partial triples go to a fixed scratch buffer of
 *   FA_DECODE_STATIC_SCRATCH_BYTES (36 MiB) compiled into libfa.so, which every
 *   GPU that loads the library holds until the process exits.  If
 *   fa_decode_workspace_size(B, H, d, n_splits) is larger than that buffer the
 *   call returns FA_ERR_UNSUPPORTED and enqueues nothing (36 MiB covers up to
 *   B·H = 2268 heads with 32 splits at d = 128).
 *   The buffer belongs to the library's decode module.  Under CUDA's default
 *   lazy module loading a device commits it (36 MiB) when it first runs any of
 *   the library's decode entry points, not when libfa.so is loaded; a caller
 *   that is about to reserve nearly all device memory should therefore make
 *   one decode call (this one, say) first.  The first call on a device also
 *   looks up the buffer's device address with that device current; make it
 *   before any stream capture begins.  The address is looked up again after a
 *   device reset gives the device a new context.
 *   Every call shares the one buffer, which keeps the last call's contents; each
 *   call rewrites every partial it reads, so nothing needs clearing.  Calls whose
 *   work overlaps on the GPU (other streams, other host threads) race on the
 *   buffer: the caller must serialise them.
 *   This entry point calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define FA_DECODE_STATIC_SCRATCH_BYTES ((size_t)36 << 20)
FA_API fa_status fa_decode_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                           int B, int H, int N_kv, int d, fa_dtype dtype, float scale,
                                           int n_splits, void* stream);

/*
 * fa_backward_workspace_size — bytes of workspace fa_backward needs:
 *   fp32 dQ accumulator B·H·N·d·4 plus per-row D and scaled LSE, 2·B·H·N·4,
 *   each part rounded up to 256.
 */
FA_API size_t fa_backward_workspace_size(int B, int H, int N, int d);

/*
 * fa_backward — gradients by recomputation.
 *   The forward kept only O and LSE; S and P are recomputed tile by tile from
 *   Q, K and LSE ("Flash Attention Backward" in the walkthrough; §二.5 of the
 *   interview notes).  The gradient itself is not on the pages; this is the
 *   textbook one for O = softmax(σQKᵀ)V:
 *     D_i = Σ_t dO_it O_it,  P = e^(S − LSE),  dV = Pᵀ dO,  dP = dO Vᵀ,
 *     dS = P ∘ (dP − D),  dQ = σ dS K,  dK = σ dSᵀ Q.
 *   q, k, v, o, dout, dq, dk, dv: [B,H,N,d] contiguous; lse [B,H,N] float32 as
 *   written by fa_forward.  workspace: at least fa_backward_workspace_size()
 *   bytes; the library clears what it needs cleared.
 *   Supported: FA_BF16, d = 64 or 128, any N >= 1 (a ragged last tile is masked).
 */
FA_API fa_status fa_backward(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                      fa_dtype dtype, float scale, void* workspace, size_t workspace_bytes,
                      void* stream);

/*
 * fa_backward_masked — fa_backward for a forward run with `mask` (FA_MASK_NONE
 *   is fa_backward).  With FA_MASK_CAUSAL (query i sees key j <= i) each key
 *   tile only visits the query tiles at or after its diagonal.  Same arguments,
 *   workspace and support as fa_backward; a causal N above 65535·128 gives
 *   FA_ERR_UNSUPPORTED.
 */
FA_API fa_status fa_backward_masked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                    const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                    fa_dtype dtype, float scale, void* workspace, size_t workspace_bytes,
                                    fa_mask mask, void* stream);

/*
 * fa_device_status — synchronises `stream`, then reports FA_ERR_DEVICE_TIMEOUT
 * if any kernel of this library has given up on a bounded pipeline wait since
 * the last call (and clears that flag), FA_ERR_CUDA on a CUDA error, else FA_OK.
 */
FA_API fa_status fa_device_status(void* stream);

/*
 * fa_watchdog_selftest — exercises the failure path of the bounded pipeline
 *   waits on the device: enqueues one CTA whose thread waits on a barrier that
 *   nothing completes.  After the wait limit (1 s) the wait gives up and
 *   records its site, exactly as a stuck pipeline would, and the kernel
 *   returns; the next fa_device_status(stream) reports FA_ERR_DEVICE_TIMEOUT
 *   ("kernel 15 gave up waiting at site 1") and clears the flag.  Nothing
 *   faults and the context stays usable.  Returns FA_OK once enqueued.
 */
FA_API fa_status fa_watchdog_selftest(void* stream);

/* Static description of a status code. */
FA_API const char* fa_status_string(fa_status s);

/* Message of the last error raised in the calling thread ("" if none). */
FA_API const char* fa_get_last_error(void);

/* Number of kernel launches this library has enqueued since it was loaded. */
FA_API uint64_t fa_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
