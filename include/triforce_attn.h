/*
 * triforce_attn.h -- C ABI of the TriForce decode-step attention library (sm_103a).
 *
 * The calls below are the data-parallel work of one hierarchical speculative
 * decoding step as described in "TriForce: Hierarchical Speculative Decoding
 * for LLMs" (section "The Architecture" / "The Three Forces of TriForce" and
 * section "Dual Rejection Sampling: Mathematical Losslessness") and in the
 * arXiv abstract of "TriForce: Lossless Acceleration of Long Sequence
 * Generation with Hierarchical Speculative Decoding":
 *   Force 1  the streaming drafter attends to attention sinks + a recent window;
 *   Force 2  the target model attends to the top-k KV blocks retrieved by
 *            key-query similarity (retrieval-sparse cache);
 *   Force 3  the target model verifies all candidates against the full cache;
 *   then each level accepts or resamples the drafted tokens losslessly.
 *
 * Conventions shared by every call
 *   - Tensor arguments are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or keeps them; it keeps no global state.
 *   - bf16 tensors are passed as uint16_t bit patterns (IEEE fp32 top half).
 *   - Layouts are dense row-major:  K, V  [B, Hkv, Lmax, D];
 *     chunk means M [B, Hkv, Cmax, D] with Cmax = ceil(Lmax / chunk);
 *     decode query q [B, Hq, D]; verify queries Q [B, Hq, T, D].
 *     Query head h reads KV head h / (Hq / Hkv) (grouped-query attention).
 *   - D must be 128 and chunk must be 8 (TF_ERR_UNSUPPORTED otherwise).
 *     Tensor pointers must be 16-byte aligned (TF_ERR_INVALID_ARG otherwise).
 *   - seq_lens [B] int32 on the device holds each sequence's valid length L_b;
 *     values are clamped to [0, Lmax].  Positions >= L_b are never read into a
 *     result (they may hold anything, including NaN).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  On error nothing is launched, except TF_ERR_CUDA,
 *     which reports a failed launch.
 *   - Workspace: calls that take `ws` need scratch of at least the size the
 *     matching *_workspace() query returns.  The buffer must be zero-filled
 *     once after allocation (cudaMemset); every call leaves its counters at
 *     zero again, so one buffer serves any sequence of calls that are ordered
 *     on the GPU.  Calls that may run concurrently need separate workspaces.
 *     Each call has its own size query, taking exactly the shape arguments
 *     the call takes, rather than one query keyed by an operation code: the
 *     sizes depend on different arguments per call, and a typed query cannot
 *     be handed the wrong ones.
 *   - Devices: every call runs on the caller's current CUDA device.  Host
 *     threads may call in concurrently, on one device or several; kernel
 *     attributes (shared-memory limits, cluster sizes) are set on each
 *     device's first call, for device ordinals below 64 (higher ordinals get
 *     an error status from the calls that need them).
 */
#ifndef TRIFORCE_ATTN_H
#define TRIFORCE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TF_API __attribute__((visibility("default")))
#else
#define TF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tf_stream_t; /* same type as cudaStream_t */

typedef enum tf_status {
  TF_OK = 0,
  TF_ERR_INVALID_ARG = 1,  /* null/misaligned pointer or inconsistent sizes; nothing launched */
  TF_ERR_UNSUPPORTED = 2,  /* valid but unsupported shape (D != 128, chunk != 8, ...) */
  TF_ERR_WORKSPACE = 3,    /* ws missing or ws_bytes below the *_workspace() size */
  TF_ERR_CUDA = 4,         /* a kernel launch failed (cudaGetLastError) */
  TF_ERR_SCRATCH_LIMIT = 5, /* the no-allocation entry point's static scratch is too small */
  TF_ERR_DEVICE_DATA = 6   /* a kernel flagged an error on the device (tf_check_status) */
} tf_status;

/* Static, human-readable text for a status code. */
TF_API const char* tf_status_string(tf_status s);

/* Library ABI version (major * 100 + minor). */
TF_API int tf_abi_version(void);

/* Device-side status of a workspace that starts with a status word (the word
 * lives in the caller's workspace, since the library keeps no state of its
 * own, so the query takes that workspace and its size): the
 * workspaces of tf_verify_attn, tf_verify_attn_tree, tf_sparse_verify_attn
 * and tf_verify_attn_offload.  Their kernels set the word when a pipeline wait
 * times out (only a hardware fault can cause that), and the outputs of every
 * call that used the workspace since then are invalid.
 * Waits for `stream` (work queued on it before this call completes first) and
 * reads the word.  Zero: returns TF_OK.  Nonzero: zeroes all ws_bytes of the
 * workspace again, in `stream` order, so the workspace can be reused, and
 * returns TF_ERR_DEVICE_DATA.  ws is device memory of ws_bytes >= 4 bytes
 * (TF_ERR_INVALID_ARG otherwise, nothing read); TF_ERR_CUDA if the copy, the
 * clearing or the wait fails.  It takes the workspace, not only the stream:
 * the library keeps no global state, so the status lives in the caller's
 * workspace. */
TF_API tf_status tf_check_status(void* ws, size_t ws_bytes, tf_stream_t stream);

/* Bounds violations recorded by the checked build of this library
 * (libtriforce_attn_debug.so, compiled with TF_DEBUG).  There every kernel
 * checks the data-dependent indices of its global-memory gathers -- cache
 * rows against [0, L_b) and Lmax, chunk-mean rows against Cmax, tensor-core
 * tiles and gathered pieces against their unit's rows, packed rows against
 * the resident buffer -- and a failed check sets a bit instead of making the
 * access: 1 cache row, 2 chunk-mean row, 4 tile or piece, 8 packed row.
 * Writes the OR of the bits recorded on the current device since the last
 * clearing to *flags (waits for the device's queued work); clear != 0 resets
 * them.  A release build returns TF_ERR_UNSUPPORTED with *flags = 0.
 * Ids outside [0, C_b) in a caller's selection are input the calls skip by
 * contract, not violations. */
TF_API tf_status tf_debug_status(uint32_t* flags, int clear);

/*
 * a1 -- chunk-mean retrieval index.
 * The retrieval-sparse cache of Force 2 selects KV blocks by key-query
 * similarity and keeps an on-demand sparse index ("The Three Forces of
 * TriForce"; "Production Advantages").  A block is `chunk` consecutive tokens,
 * represented by the mean of its keys:
 *   M[b,g,c,:] = bf16_round_nearest_even( (1/n_c) * sum_{t in chunk c, t < L_b} K[b,g,t,:] )
 * with n_c the number of valid tokens of chunk c (8, fewer for the last partial
 * chunk).  Chunks with no valid token are written as zeros.  Only chunks
 * c_begin <= c < c_end are written (0 <= c_begin <= c_end <= Cmax), so a
 * decode step can refresh just the chunk that changed.
 * The mean is rounded once: the sum is carried as an unevaluated pair of fp32
 * values, exact for any eight bf16 values whose magnitudes span < 2^40.
 */
TF_API tf_status tf_build_chunk_means(const uint16_t* K, const int32_t* seq_lens,
                               int B, int Hkv, int Lmax, int D, int chunk,
                               int c_begin, int c_end,
                               uint16_t* M, tf_stream_t stream);

/*
 * a2 + a3 -- chunk scores and top-k selection (Force 2 retrieval).
 * Score of chunk c for (b, g): s = sum_d (sum_{h in group g} q[b,h,d]) * M[b,g,c,d],
 * accumulated in fp32 (no softmax scale: it does not change the order).
 * Selection keeps the kc highest-scoring chunks among C_b = ceil(L_b / chunk);
 * equal scores go to the lower chunk id; output ids are ascending.
 *   idx   [B, Hkv, kc] int32   selected chunk ids, slots >= n_sel hold -1
 *   n_sel [B, Hkv]     int32   min(kc, C_b)
 *   s_cut [B, Hkv]     float   smallest selected score (nullable; -inf if none)
 * Scores must be finite (NaN scores rank above every number).  Contexts up to
 * 8 x 16384 chunks (1,048,576 tokens) per sequence.
 * Workspace: none; tf_chunk_scores_topk_workspace() returns 0 and ws may be
 * NULL (scores and the selection stay in on-chip shared memory of one
 * thread-block cluster per (b, g)).
 */
TF_API size_t tf_chunk_scores_topk_workspace(int B, int Hkv, int Lmax, int chunk);
TF_API tf_status tf_chunk_scores_topk(const uint16_t* q, const uint16_t* M, const int32_t* seq_lens,
                               int B, int Hq, int Hkv, int Lmax, int D, int chunk, int kc,
                               int32_t* idx, int32_t* n_sel, float* s_cut,
                               void* ws, size_t ws_bytes, tf_stream_t stream);

/*
 * a4 (+ a5) -- retrieval-sparse decode attention (Force 2).
 * For query head h of group g:  out[b,h,:] = softmax(scale * q_h . K_S) V_S
 * where S is the valid tokens (t < L_b) of the chunks idx[b,g,0:n_sel[b,g]].
 * Ids outside [0, C_b) are skipped; a repeated id is attended once per
 * occurrence.  An empty set gives a zero output row.  fp32 accumulation,
 * split over the selected chunks and merged with the log-sum-exp identity.
 *   out [B, Hq, D] float32
 * Workspace: tf_sparse_decode_attn_workspace(B, Hq, Hkv, kc) bytes.
 */
TF_API size_t tf_sparse_decode_attn_workspace(int B, int Hq, int Hkv, int kc);
TF_API tf_status tf_sparse_decode_attn(const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                const int32_t* seq_lens, const int32_t* idx, const int32_t* n_sel,
                                int B, int Hq, int Hkv, int Lmax, int D, int chunk, int kc,
                                float scale, float* out,
                                void* ws, size_t ws_bytes, tf_stream_t stream);

/*
 * tf_sparse_decode_attn without a workspace, for callers that cannot allocate
 * device memory (the paper has no counterpart; this is a deployment aid).
 * Some hosts cannot call cudaMalloc: an engine that owns every device
 * allocation, a plugin loaded into such an engine, or a latency-critical loop
 * where allocating (and the synchronisation it may bring) is not allowed.
 * Same inputs and outputs as tf_sparse_decode_attn.  The result agrees with
 * tf_sparse_decode_attn within the attention tolerance (max abs error 2e-3),
 * not bit for bit: this call always runs the CUDA-core gather kernel, while
 * tf_sparse_decode_attn runs the tensor-core kernel for groups of two or more
 * query heads per KV head (at 128K, batch 4 x 8 KV heads x 4 heads per group,
 * about 50 us per call here against about 30 us there).
 * The split-K scratch is a 32 MiB file-scope device array instead of `ws`,
 * held by every GPU that loads this library until the process exits.  The
 * tickets use its first 64 KiB and the partial results the rest: a problem
 * fits when its partials need at most 32 MiB - 64 KiB, i.e. at kc = 512 up to
 * B * Hkv = 499 (one query head per KV head), 249 (two), 124 (three or four,
 * e.g. batch 8 x 8 KV heads x 4 heads per group: 17.2 MB) or 62 (five to
 * eight).  Larger problems return TF_ERR_SCRATCH_LIMIT without launching.
 * The first successful call on each device sets up that device's copy (looks
 * up its address with cudaGetSymbolAddress and zeroes the ticket area with a
 * synchronous cudaMemset), so make it before any stream capture: on a stream
 * that is being captured it returns TF_ERR_INVALID_ARG without touching the
 * device, and a set-up that failed is tried again on the next call.  All
 * calls share the one array and leave their contents in it: calls that may
 * overlap on the GPU (unordered streams) race and give wrong results.  It
 * allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
TF_API tf_status tf_sparse_decode_attn_noalloc(const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                const int32_t* seq_lens, const int32_t* idx, const int32_t* n_sel,
                                int B, int Hq, int Hkv, int Lmax, int D, int chunk, int kc,
                                float scale, float* out, tf_stream_t stream);

/*
 * a2 + a3 + a4 (+ a5) fused -- the whole Force 2 retrieval drafter step of one
 * layer in one launch ("TriForce: Hierarchical Speculative Decoding for LLMs",
 * "The Three Forces of TriForce": attention over only the KV blocks of highest
 * key-query similarity, within a fixed budget).  Computes exactly what
 * tf_chunk_scores_topk followed by tf_sparse_decode_attn compute:
 *   idx, n_sel, s_cut  as tf_chunk_scores_topk (s_cut may be NULL);
 *   out [B, Hq, D] float32  as tf_sparse_decode_attn over that selection.
 * Scores, the selection and the split-K partial states stay on chip (one
 * thread-block cluster per (b, g)), so there is no workspace.  Limits:
 * kc <= 2048, Hq / Hkv <= 4, contexts up to 8 x 16384 chunks, and for
 * Hq / Hkv >= 2 (chunks loaded by TMA) B * Hkv * Lmax < 2^31 (else
 * TF_ERR_UNSUPPORTED; the two separate calls have no such limits).  Device
 * pointers, 16-byte aligned q, M, K, V and out.
 */
TF_API tf_status tf_retrieval_draft_attn(const uint16_t* q, const uint16_t* M, const uint16_t* K,
                                  const uint16_t* V, const int32_t* seq_lens,
                                  int B, int Hq, int Hkv, int Lmax, int D, int chunk, int kc,
                                  float scale, int32_t* idx, int32_t* n_sel, float* s_cut,
                                  float* out, tf_stream_t stream);

/*
 * tf_retrieval_draft_attn with a lower bound on each (b, g)'s cut score, e.g.
 * the s_cut of the previous decode step lowered by a margin.  cut_hint
 * [B, Hkv] float32, device, required (NaN in a slot: no bound for that
 * (b, g)).  The outputs are exactly those of tf_retrieval_draft_attn on the
 * same inputs, whatever the bounds: idx, n_sel and s_cut bit for bit, out up
 * to the fp32 summation order.  Only the time changes.  When between kc and
 * 4096 chunks of the (b, g) score at least the bound (and no CTA of its
 * cluster holds more than 2048 of them), the cut is found from those keys
 * alone: one cluster barrier and a gather of those keys replace the
 * cluster-wide histogram round and the second barrier of the unhinted path.
 * Otherwise (a bound above the cut, or one that admits too many chunks) the
 * count exchange is the only extra cost and the unhinted path runs.  A launch
 * takes as long as its slowest (b, g), so the bound pays when it holds on
 * every (b, g): 0.7 x the previous step's s_cut did on every one in the
 * synthetic decode steps measured here.  Same limits as
 * tf_retrieval_draft_attn.
 */
TF_API tf_status tf_retrieval_draft_attn_hinted(const uint16_t* q, const uint16_t* M, const uint16_t* K,
                                                const uint16_t* V, const int32_t* seq_lens, int B, int Hq,
                                                int Hkv, int Lmax, int D, int chunk, int kc, float scale,
                                                const float* cut_hint, int32_t* idx, int32_t* n_sel,
                                                float* s_cut, float* out, tf_stream_t stream);

/*
 * a2 + a3 + a4 and a6 in one launch, for GQA groups (2 <= Hq / Hkv <= 4):
 * tf_retrieval_draft_attn (cut_hint as tf_retrieval_draft_attn_hinted; NULL:
 * no bound) plus tf_stream_window_attn of the same decode queries q over the
 * same cache ("TriForce: Hierarchical Speculative Decoding for LLMs", "The
 * Three Forces of TriForce": Force 1's sinks + recent window and Force 2's
 * retrieved blocks, both drafters' attention for the same token).  The
 * window's keys, [0, min(n_sink, L)) and [max(n_sink, L - window), L), enter
 * the drafter's chunk lists as 8-row pieces, and its rows ride in the spare
 * rows of the drafter's tensor-core fragments, so the window needs no launch
 * of its own.  Outputs: idx, n_sel, s_cut, out as tf_retrieval_draft_attn;
 * wout [B, Hq, 128] fp32 as tf_stream_window_attn (within the attention
 * tolerance).  Limits: those of tf_retrieval_draft_attn, Hq / Hkv from 2 to
 * 4, and kc + ceil(n_sink / 8) + ceil(window / 8) + 1 <= 2048 (else
 * TF_ERR_UNSUPPORTED).  Errors: NULL or misaligned wout, negative n_sink or
 * window -> TF_ERR_INVALID_ARG; otherwise as tf_retrieval_draft_attn.
 */
TF_API tf_status tf_retrieval_window_draft_attn(const uint16_t* q, const uint16_t* M, const uint16_t* K,
                                  const uint16_t* V, const int32_t* seq_lens,
                                  int B, int Hq, int Hkv, int Lmax, int D, int chunk, int kc,
                                  float scale, const float* cut_hint, int n_sink, int window,
                                  int32_t* idx, int32_t* n_sel, float* s_cut, float* out,
                                  float* wout, tf_stream_t stream);

/*
 * Level-1 verification over the retrieval cache:
 * the retrieval drafter -- the target model over the retrieved KV blocks --
 * checks the tiny drafter's candidates in one pass ("TriForce: Hierarchical
 * Speculative Decoding for LLMs", "The Three Forces of TriForce" and "Dual
 * Rejection Sampling: Mathematical Losslessness").  The cache already holds
 * the T candidates' keys/values at positions L-T .. L-1; query j
 * (0 <= j < T) of head h in group g sees the valid tokens (t < L) of the
 * chunks idx[b,g,0:n_sel[b,g]] that lie before the candidates (t < L-T), and
 * candidates 0..j (t in [L-T, L-T+j]):
 *   out[b,h,j,:] = softmax(scale * Q[b,h,j] . K_P) V_P     (float32)
 * Ids outside [0, C_b) are skipped; a repeated id is attended once per
 * occurrence.  Q [B, Hq, T, D] bf16, out [B, Hq, T, D] float32, 1 <= T <= 16.
 * Tensor-core kernel (tcgen05, bf16 in, fp32 accumulate): each 128-key tile is
 * gathered from sixteen 8-row pieces by TMA.  Workspace:
 * tf_sparse_verify_attn_workspace(B, Hq, Hkv, kc, T) bytes, zeroed once; its
 * first int is a status word (nonzero after a device-side timeout).
 */
TF_API size_t tf_sparse_verify_attn_workspace(int B, int Hq, int Hkv, int kc, int T);
TF_API tf_status tf_sparse_verify_attn(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                                const int32_t* seq_lens, const int32_t* idx, const int32_t* n_sel,
                                int B, int Hq, int Hkv, int Lmax, int D, int chunk, int kc, int T,
                                float scale, float* out, void* ws, size_t ws_bytes, tf_stream_t stream);

/*
 * a6 (+ a5) -- StreamingLLM sink + window attention (Force 1 drafter).
 * Positions P = [0, min(n_sink, L)) U [max(n_sink, L - window), L): the first
 * n_sink tokens plus the most recent `window` tokens, de-duplicated.
 *   out [B, Hq, D] float32 = softmax(scale * q_h . K_P) V_P
 * Workspace: tf_stream_window_attn_workspace(B, Hq, Hkv, n_sink, window) bytes.
 */
TF_API size_t tf_stream_window_attn_workspace(int B, int Hq, int Hkv, int n_sink, int window);
TF_API tf_status tf_stream_window_attn(const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                const int32_t* seq_lens,
                                int B, int Hq, int Hkv, int Lmax, int D, int n_sink, int window,
                                float scale, float* out,
                                void* ws, size_t ws_bytes, tf_stream_t stream);

/*
 * a7 (+ a5) -- full-cache verification attention (Force 3).
 * The cache already holds the T candidates' keys/values at positions
 * L-T .. L-1 and the candidates form a chain, so verify query j (0 <= j < T)
 * attends to positions [0, L - T + j]:
 *   out[b,h,j,:] = softmax(scale * Q[b,h,j] . K_{0..L-T+j}) V_{0..L-T+j}
 * Rows with no visible position (L - T + j < 0) are zero.  1 <= T <= 16;
 * B * Hkv * Lmax < 2^31.  Tensor-core kernel: K and V tiles stream in by TMA,
 * S = K Q^T and O = P V run as tcgen05 MMAs (bf16 in, fp32 accumulate; the
 * softmax weights P enter P V as bf16 hi + lo parts, P = hi + lo to 2^-17, and
 * the row sums use the fp32 weights).
 *   out [B, Hq, T, D] float32
 * Workspace: tf_verify_attn_workspace(B, Hq, Hkv, Lmax, T) bytes.  Its first
 * int32 is a status word: nonzero means a pipeline wait timed out (which only a
 * hardware fault can cause) and the output is invalid; re-zero the workspace
 * before reusing it.
 */
TF_API size_t tf_verify_attn_workspace(int B, int Hq, int Hkv, int Lmax, int T);
TF_API tf_status tf_verify_attn(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                         const int32_t* seq_lens,
                         int B, int Hq, int Hkv, int Lmax, int D, int T,
                         float scale, float* out,
                         void* ws, size_t ws_bytes, tf_stream_t stream);

/*
 * a7 and a6 in one call: tf_verify_attn plus tf_stream_window_attn for the
 * decode queries q [B, Hq, 128] bf16 over the same cache ("TriForce:
 * Hierarchical Speculative Decoding for LLMs", "The Three Forces of
 * TriForce": Force 1's attention sinks plus recent window, Force 3's check of
 * the candidates against the full cache).  With G = Hq / Hkv, when the G
 * window rows of a KV head fill padding rows of the verify kernel (the
 * G*(T+1) rows need neither more 32-row groups nor a wider group, rounded up
 * to 8 rows, than the G*T candidate rows: G = 1 with T = 6, G = 4 with
 * T = 5; not G = 1 with T = 8, G = 4 with T = 6 nor G = 8 with T = 4), they
 * ride as extra query rows of the verify launch, masked to the keys
 * [0, min(n_sink, L)) and [max(n_sink, L - window), L): one launch, the
 * cache read once.  Otherwise the call makes two launches on the stream
 * (tf_stream_window_attn, then tf_verify_attn): a wider kernel or a group of
 * window rows alone costs more than the window launch.
 * out [B, Hq, T, 128] as tf_verify_attn, wout [B, Hq, 128] as
 * tf_stream_window_attn (both fp32, within the attention tolerance of the
 * separate calls).  Workspace from tf_verify_window_attn_workspace (0 for
 * arguments it refuses); its status word sits where tf_verify_attn's does.
 * T <= 16.  Device pointers, 16-byte aligned.  Errors: null pointer,
 * negative size, n_sink or window, Hq % Hkv != 0 or misalignment ->
 * TF_ERR_INVALID_ARG; D != 128 or T > 16 -> TF_ERR_UNSUPPORTED; a workspace
 * below the size -> TF_ERR_WORKSPACE; all before any launch.
 */
TF_API size_t tf_verify_window_attn_workspace(int B, int Hq, int Hkv, int Lmax, int T, int n_sink, int window);
TF_API tf_status tf_verify_window_attn(const uint16_t* Q, const uint16_t* q, const uint16_t* K,
                                       const uint16_t* V, const int32_t* seq_lens, int B, int Hq, int Hkv,
                                       int Lmax, int D, int T, int n_sink, int window, float scale,
                                       float* out, float* wout, void* ws, size_t ws_bytes, tf_stream_t stream);

/*
 * a7 over a candidate tree ("TriForce: Hierarchical Speculative Decoding for
 * LLMs", "The Three Forces of TriForce": Force 2
 * arranges the surviving candidates as a tree and Force 3 checks the whole
 * tree in one forward pass with tree attention).  The T candidates sit at
 * positions L-T .. L-1 as for tf_verify_attn; parent[b*T + j] (device int32,
 * [B, T]) is the candidate that candidate j extends, or -1 when j extends the
 * prefix directly.  Query j attends to the prefix [0, L-T) and to candidate j
 * and its ancestors:
 *   out[b,h,j,:] = softmax(scale * Q[b,h,j] . K_P) V_P,
 *   P = [0, L-T) U { L-T+i : i = j, parent(j), parent(parent(j)), ... }
 * parent = j - 1 for every j is the chain of tf_verify_attn (same result).  A
 * parent outside [-1, j) ends the ancestor walk there (it is read as -1).
 * Same shapes, workspace and errors as tf_verify_attn; parent may not be null.
 */
TF_API tf_status tf_verify_attn_tree(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                              const int32_t* seq_lens, const int32_t* parent,
                              int B, int Hq, int Hkv, int Lmax, int D, int T,
                              float scale, float* out,
                              void* ws, size_t ws_bytes, tf_stream_t stream);

/* Resident retrieval cache: the rows the retrieval drafter attends to, packed
 * into a buffer of their own ("TriForce: Lossless Acceleration of Long
 * Sequence Generation with Hierarchical Speculative Decoding", "Abstract
 * (arXiv)": the retrieval-sparse cache is the middle draft level and, when
 * offloading, the full cache lives in host memory; project summary, "How It
 * Works").  For each (b, g) the valid tokens (t < L_b) of the chunks
 * idx[b,g,0:n_sel[b,g]] are copied in list order to rows 0.. of
 *   Kc, Vc [B, Hkv, kc * chunk, D]   (device memory; rows at and past the
 *                                      packed count are not written)
 *   lens [B * Hkv] int32              packed rows of each (b, g)
 *   n_chunks [B * Hkv] int32          ceil(lens / chunk)
 * Ids outside [0, C_b) add no rows; a repeated id is copied once per
 * occurrence; n_sel is clamped to [0, kc].  K, V [B, Hkv, Lmax, D] are device
 * memory of the current device or host memory the CUDA runtime pinned or
 * registered (read over the host link); any other pointer is refused with
 * TF_ERR_INVALID_ARG before launch.  kc <= 4096.
 * The packed buffer is attended through tf_sparse_decode_attn viewed as B*Hkv
 * sequences of one KV head each: q [B*Hkv, G, D], K/V [B*Hkv, 1, kc*chunk, D],
 * seq_lens = lens, idx[u, 0, i] = i and n_sel = n_chunks, which gives the
 * attention over the original selection. */
TF_API tf_status tf_pack_retrieval_cache(const uint16_t* K, const uint16_t* V, const int32_t* seq_lens,
                                  const int32_t* idx, const int32_t* n_sel, int B, int Hkv, int Lmax,
                                  int D, int chunk, int kc, uint16_t* Kc, uint16_t* Vc, int32_t* lens,
                                  int32_t* n_chunks, tf_stream_t stream);

/*
 * a7 with the cache offloaded to host memory ("TriForce: Lossless Acceleration
 * of Long Sequence Generation with Hierarchical Speculative Decoding",
 * "Abstract (arXiv)": the whole cache is read for every generated token;
 * project summary, "Highlighted Details" / "How It Works": the original
 * offloads the cache to CPU memory).  Computes exactly what tf_verify_attn
 * computes; only where K and V live differs.
 *   K_host, V_host: [B, Hkv, Lmax, D] bf16 in host memory (pinned, so that the
 *     copies run asynchronously at full link rate; pageable memory works but
 *     copies synchronously).  Q, seq_lens, out and ws are device memory.
 *   L_stream: positions [0, L_stream) are streamed; every seq_lens[b] must be
 *     <= L_stream <= Lmax (lengths are clamped to L_stream).
 *   seg_rows: positions per segment.  Segment s (positions [s * seg_rows,
 *     (s + 1) * seg_rows)) is copied on copy_stream into one of two device
 *     staging slots (one 2-D copy per tensor: every (b, g) unit's rows) while
 *     the previous segment is attended on `stream`; each segment leaves every
 *     query row's (max, row sum, unnormalised O) in the workspace and one
 *     final kernel merges them (log-sum-exp identity).
 *   Ordering: work queued on `stream` before the call completes before the
 *   first copy; `out` is ready in `stream` order.  copy_stream may equal
 *   stream (no overlap).
 * Workspace: tf_verify_attn_offload_workspace(B, Hq, Hkv, Lmax, T, seg_rows)
 * bytes, zeroed once before first use; its first int32 is the status word of
 * tf_verify_attn.  Errors: TF_ERR_INVALID_ARG / UNSUPPORTED / WORKSPACE before
 * any work is queued; TF_ERR_CUDA if a copy or launch fails.
 */
TF_API size_t tf_verify_attn_offload_workspace(int B, int Hq, int Hkv, int Lmax, int T, int seg_rows);
TF_API tf_status tf_verify_attn_offload(const uint16_t* Q, const uint16_t* K_host, const uint16_t* V_host,
                                 const int32_t* seq_lens, int L_stream, int B, int Hq, int Hkv, int Lmax,
                                 int D, int T, float scale, float* out, int seg_rows, void* ws,
                                 size_t ws_bytes, tf_stream_t stream, tf_stream_t copy_stream);

/*
 * a8 -- lossless speculative accept / resample of one verification level
 * ("Dual Rejection Sampling: Mathematical Losslessness").
 * With p_i = softmax(tgt_logits[b,i,:] / temperature) (the verifier) and
 * q_i = softmax(drf_logits[b,i,:] / temperature) (the drafter), drafted token
 * x_i is accepted when u_acc[b,i] <= p_i(x_i) / q_i(x_i) (always when
 * q_i(x_i) == 0).  At the first rejection j the next token is drawn from
 * max(0, p_j - q_j) normalised (from p_j if that residual is all zero); if
 * all g drafted tokens are accepted, a bonus token is drawn from p_g.  Draws
 * use the index-order inverse CDF with u_res[b]: the first t whose cumulative
 * weight exceeds u_res * total.
 * The same call serves both levels of the hierarchy: tiny drafter -> retrieval
 * drafter, then retrieval drafter -> target (pass the first level's
 * out_tokens as the second level's drf_tokens).
 *   tgt_logits [B, gamma+1, V] f32, drf_logits [B, gamma, V] f32
 *   drf_tokens [B, gamma] int32; an entry outside [0, V) ends the draft
 *   u_acc [B, gamma] f32, u_res [B] f32, uniforms in [0, 1)
 *   n_acc [B] int32 (accepted count), next_token [B] int32
 *   out_tokens [B, gamma+1] int32 (nullable): accepted drafts, next token, -1 pad
 *     (an output beyond n_acc and next_token so that the second level can take
 *     the first level's result directly as its draft, with no host step)
 * temperature > 0.  gamma >= 0, V >= 1.  Probabilities use fp32 exponentials,
 * normalisers summed in fp32 then fp64, an fp64 ratio test, and cumulative
 * sums carried as exact fp32 pairs (fp64 for a warp-sized vocabulary), so a
 * decision can differ from exact arithmetic only when a uniform lies within
 * ~1e-6 of its boundary.
 * Workspace: tf_spec_accept_workspace(B, gamma) bytes (per-row normalisers;
 * needs no zeroing).  Two kernel launches.
 */
TF_API size_t tf_spec_accept_workspace(int B, int gamma);
TF_API tf_status tf_spec_accept(const float* tgt_logits, const float* drf_logits, const int32_t* drf_tokens,
                         const float* u_acc, const float* u_res,
                         int B, int gamma, int V, float temperature,
                         int32_t* n_acc, int32_t* next_token, int32_t* out_tokens,
                         void* ws, size_t ws_bytes, tf_stream_t stream);

/*
 * a8 over a candidate tree ("TriForce: Hierarchical Speculative Decoding for
 * LLMs", "The Three Forces of TriForce": Force 2 arranges the candidates as a
 * tree and Force 3 verifies the tree in one pass with the speculative
 * rejection rule; "Dual Rejection Sampling: Mathematical Losslessness": the
 * per-candidate test and residual).  The pages print no rule for several
 * candidates extending one node; this call applies the printed rule to them
 * one at a time: the children of a node, drawn independently from the
 * drafter's distribution there, are tested in index order against the
 * current target p' (at first the verifier's distribution at the node); a
 * child is kept when u_acc <= p'(x) / q(x) (always when q(x) == 0) and the
 * walk goes on at it with the verifier's distribution after it; a child that
 * fails replaces p' by max(0, p' - q) normalised (p' is kept when that
 * residual is all zero) and its next sibling is tested.  When the current
 * node has no child left, the next token is drawn from p' with the
 * index-order inverse CDF of tf_spec_accept (u_res): the residual after the
 * last rejection, or the bonus token from the verifier row after the node.
 * With parent[j] = j - 1 this is tf_spec_accept, decision for decision.
 *   tgt_logits [B, T+1, V] f32: row 0 the verifier at the prefix, row 1+j the
 *     verifier after candidate j (as tf_verify_attn_tree's query j gives it)
 *   drf_logits [B, T, V] f32: row j the drafter distribution candidate j was
 *     drawn from (its parent's; siblings share it)
 *   drf_tokens [B, T] int32: an entry outside [0, V) removes the candidate and
 *     its subtree
 *   parent [B, T] int32: the candidate that j extends, -1 for the prefix; a
 *     link outside [-1, j) is read as -1 (as in tf_verify_attn_tree)
 *   u_acc [B, T] f32 (the uniform of candidate j's test), u_res [B] f32
 *   n_acc [B] int32: depth of the kept path; next_token [B] int32
 *   out_tokens [B, T+1] int32 (nullable): kept tokens, next token, -1 pad
 *   acc_nodes [B, T] int32 (nullable): indices of the kept candidates, -1 pad
 * T >= 0 (drf_logits, drf_tokens, parent and u_acc may be NULL when T == 0),
 * V >= 1, temperature > 0.  Precision as tf_spec_accept; p' after a rejection
 * is held as fp32 weights.  Workspace: tf_spec_accept_tree_workspace(B, T, V)
 * bytes (normalisers and two vocabulary rows per sequence; needs no zeroing).
 * Two kernel launches; a rejection costs one pass over the vocabulary.
 */
TF_API size_t tf_spec_accept_tree_workspace(int B, int T, int V);
TF_API tf_status tf_spec_accept_tree(const float* tgt_logits, const float* drf_logits, const int32_t* drf_tokens,
                              const int32_t* parent, const float* u_acc, const float* u_res,
                              int B, int T, int V, float temperature,
                              int32_t* n_acc, int32_t* next_token, int32_t* out_tokens, int32_t* acc_nodes,
                              void* ws, size_t ws_bytes, tf_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TRIFORCE_ATTN_H */
