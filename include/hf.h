/*
 * hf.h -- C ABI of the hybrid attention step of Hybrid Forcing
 * ("Long-Horizon Streaming Video Generation via Hybrid Attention with
 * Decoupled Distillation"), for NVIDIA B300 (sm_103a).
 *
 * The step has two paths whose outputs are summed (Spanish technical
 * summary, section 2.A, "Atención Híbrida": the final output is the sum of
 * the compressed linear history and the sparse local attention):
 *   - block-sparse sliding-window softmax attention: query and key blocks
 *     are mean-pooled and scored, and every query block attends only to its
 *     top-K key blocks of the window (English technical summary, section
 *     2.A.2 "Block-Sparse Sliding Window Attention");
 *   - linear temporal attention: a read of a constant-size per-head state
 *     S = sum phi(k) v^T, z = sum phi(k) that absorbs every frame evicted
 *     from the window (English technical summary, section 2.A.1 "Linear
 *     Temporal Attention"; arXiv abstract: "a compact key-value state to
 *     incrementally absorb evicted tokens").  phi(x) = elu(x) + 1.
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless marked (host).  The caller owns
 *     every buffer, including the workspace; the library never allocates or
 *     frees device memory.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All work is enqueued on it; nothing synchronises except
 *     hf_get_device_status.
 *   - Argument errors are returned synchronously before anything is
 *     launched (HF_ERR_INVALID_ARG / HF_ERR_UNSUPPORTED).  A failed launch
 *     returns HF_ERR_CUDA.  A kernel that gives up waiting (every wait in
 *     every kernel is bounded) records HF_ERR_TIMEOUT in the workspace
 *     status word, which hf_get_device_status reads.  hf_last_error() gives a
 *     one-line description of the last error on the calling thread.
 *   - All device pointers must be 16-byte aligned (TMA requirement).
 *   - Results are deterministic: no floating-point atomics, fixed
 *     reduction orders.
 *
 * Shapes (b = batch, H = heads, d = head_dim, N_f = tokens per latent
 * frame, C = chunk frames, W = window frames INCLUDING the chunk,
 * beta = block size, bpf = ceil(N_f / beta)):
 *   Q      bf16 [b, H, C*N_f, d]         the chunk's queries (frames in order)
 *   Kc, Vc bf16 [b, H, W, slot_stride, d] ring of W frame slots, slot_stride >= N_f
 *   slot_map (host) int32 [n_win]        logical window frame w (0 = oldest,
 *                                        the last C are the chunk) -> ring slot
 *   S      fp32 [b, H, d, d]             row = feature of phi(k), column = value channel
 *   z      fp32 [b, H, d]
 *   nQB = C*bpf query blocks, nKB = n_win*bpf key blocks, K_eff = min(topk, nKB)
 *   Blocks tile every frame separately from its first token; the last block
 *   of a frame holds N_f - (bpf-1)*beta tokens.  Key block kb = w*bpf + j.
 */
#ifndef HF_H
#define HF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HF_ABI_VERSION 3

#if defined(__GNUC__)
#define HF_API __attribute__((visibility("default")))
#else
#define HF_API
#endif

/* Limits checked on entry (HF_ERR_UNSUPPORTED beyond them). */
#define HF_MAX_WINDOW_FRAMES 64
#define HF_MAX_KEY_BLOCKS 1024

typedef enum {
    HF_OK = 0,
    HF_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, inconsistent sizes */
    HF_ERR_UNSUPPORTED = 2,   /* valid but outside the supported shapes */
    HF_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    HF_ERR_TIMEOUT = 4,       /* a kernel's bounded wait ran out (device status) */
    HF_ERR_DEVICE_CHECK = 5   /* a kernel found an inconsistent input (device status) */
} hf_status;

typedef struct {
    int32_t batch;            /* >= 1 */
    int32_t heads;            /* >= 1 */
    int32_t head_dim;         /* 64 or 128 */
    int32_t tokens_per_frame; /* N_f >= 1 */
    int32_t window_frames;    /* W, includes the current chunk; 1..HF_MAX_WINDOW_FRAMES */
    int32_t chunk_frames;     /* C, 1..W */
    int32_t block_size;       /* beta: 32, 64 or 128 */
    int32_t topk;             /* K >= 1; clamped to nKB */
    float softmax_scale;      /* 0 -> 1/sqrt(head_dim) */
    float lin_eps;            /* added to the linear-read denominator; e.g. 1e-6 */
} hf_config;

/* Version of this ABI (HF_ABI_VERSION). */
HF_API int32_t hf_abi_version(void);

/* Text for a status code (static storage). */
HF_API const char *hf_status_string(hf_status s);

/* One-line description of the last error returned on this thread. */
HF_API const char *hf_last_error(void);

/* Workspace bytes the forward/scoring/attention/absorb calls need for
 * `cfg` (sized for a full window of cfg->window_frames frames).  The same
 * workspace may be reused by every call on one stream; calls that run
 * concurrently need separate workspaces.  Calls that share one may differ
 * in topk (up to cfg->topk of the sizing call) and in the window, not in the
 * other fields.  It must be zeroed once before first use (its first 256
 * bytes are the device status word, read and cleared by
 * hf_get_device_status).  The counters that the attention kernel keeps for
 * tile pairs it splits between CTAs follow; every forward resets them before
 * its attention kernel runs, so a call that gave up part-way (a device
 * error) leaves nothing behind that changes a later call.  The workspace
 * also holds the pooled-key cache of the layer's ring (see hf_pool_keys) and
 * the state as the linear read's tensor-core operand (see
 * HF_FWD_STATE_PREPARED), at offsets that do not depend on topk: one
 * workspace per ring and state. */
HF_API hf_status hf_workspace_size(const hf_config *cfg, size_t *bytes /* host */);

/* S = 0, z = 0 (the empty state). */
HF_API hf_status hf_state_reset(const hf_config *cfg, float *S, float *z, void *stream);

/* Absorb evicted frames into the state (English technical summary, section
 * 2.A.1: the state incrementally aggregates evicted frames):
 *   S += sum_t phi(K_ev[t]) V_ev[t]^T,  z += sum_t phi(K_ev[t])
 * for every (batch, head).  K_ev, V_ev: bf16 [b, H, n_ev_tokens, d].
 * n_ev_tokens = 0 is a no-op.  tcgen05 GEMM with fp32 accumulation; phi(k)
 * enters the MMA as a bf16 hi + lo pair, so S carries ~fp32 accuracy.  The
 * new S is also written to the workspace as the linear read's tensor-core
 * operand (see HF_FWD_STATE_PREPARED). */
HF_API hf_status hf_absorb_evicted(const hf_config *cfg, float *S, float *z,
                            const uint16_t *K_ev, const uint16_t *V_ev,
                            int32_t n_ev_tokens, void *ws, void *stream);

/* Flag of hf_absorb_evicted_strided. */
#define HF_ABSORB_SHARE_SMS 1u

/* The same as hf_absorb_evicted, for evicted tokens that are not packed per
 * head: token t of head h is the row at K_ev + (h * head_stride_tokens + t) * d
 * (and likewise for V_ev), with head_stride_tokens >= n_ev_tokens.  This
 * absorbs frames straight out of the key/value ring (frames contiguous in
 * their slots, slot_stride = N_f) without a copy.  flags: 0, or
 * HF_ABSORB_SHARE_SMS when the absorb runs beside other kernels (the next
 * chunk's key pooling and the forward's prologue, on another stream): it then
 * keeps fewer tiles in flight on about half of the SMs, so that those kernels fit
 * beside it.  The state then differs from the other mode's only in the order
 * of one fp32 reduction (a few ulps); each mode is deterministic. */
HF_API hf_status hf_absorb_evicted_strided(const hf_config *cfg, float *S, float *z,
                                           const uint16_t *K_ev, const uint16_t *V_ev,
                                           int32_t n_ev_tokens, int64_t head_stride_tokens,
                                           void *ws, void *stream, uint32_t flags);

/* Block importance scores (English technical summary, section 2.A.2):
 *   scores[b,h,qb,kb] = <mean(Q block qb), mean(K block kb)>  (float32)
 * Means are sequential float32 sums in token order divided by the token
 * count; the dot is a sequential fused multiply-add chain over channels in
 * ascending order; -0 becomes +0.  This fixed arithmetic makes the scores,
 * and so the selected indices, bit-reproducible.
 * scores: fp32 [b, H, nQB, nKB].  C <= n_win <= W. */
HF_API hf_status hf_block_scores(const hf_config *cfg, const uint16_t *Q, const uint16_t *Kc,
                          int32_t slot_stride, const int32_t *slot_map /* host */,
                          int32_t n_win, float *scores, void *ws, void *stream);

/* Top-K key blocks per query block (English technical summary, section
 * 2.A.2: only the top-K most informative blocks are kept).  Order: score
 * descending, then block index ascending (ties go to the lower index);
 * the K_eff = min(topk, nKB) winners are written in ascending index order.
 * scores: fp32 [b, H, nQB, nKB] (finite); idx: int32 [b, H, nQB, K_eff]. */
HF_API hf_status hf_topk_blocks(const hf_config *cfg, const float *scores, int32_t nQB, int32_t nKB,
                         int32_t *idx, void *stream);

/* Block-sparse softmax attention (English technical summary, section
 * 2.A.2): for every query token, softmax(scale * q.k) over the tokens of
 * the key blocks selected for its query block, times V.  No other mask.
 * idx: int32 [b, H, nQB, K_eff] ascending (as written by hf_topk_blocks).
 * O_swa: fp32 [b, H, C*N_f, d].  tcgen05 MMAs, bf16 operands, fp32
 * accumulation and softmax. */
HF_API hf_status hf_sparse_swa_attn(const hf_config *cfg, const uint16_t *Q, const uint16_t *Kc,
                             const uint16_t *Vc, int32_t slot_stride,
                             const int32_t *slot_map /* host */, int32_t n_win,
                             const int32_t *idx, float *O_swa, void *ws, void *stream);

/* Linear read (English technical summary, section 2.A.1):
 *   o_lin = phi(q)^T S / (phi(q)^T z + lin_eps)   (float32)
 * O: fp32 [b, H, C*N_f, d]; accumulate != 0 adds o_lin to O, else stores. */
HF_API hf_status hf_linear_read(const hf_config *cfg, const uint16_t *Q, const float *S,
                         const float *z, float *O, int32_t accumulate, void *stream);

/* The whole hybrid attention step for one chunk (both paths, summed; Spanish
 * technical summary, section 2.A): pooling, scores, top-K, block-sparse
 * attention and, fused into its epilogue, the linear read and the sum.
 *   O = bf16( o_swa + o_lin )   bf16 [b, H, C*N_f, d], round to nearest even
 * idx_out (optional, may be NULL): int32 [b, H, nQB, K_eff].
 * S, z: the state AFTER absorbing the frames this chunk evicted. */
HF_API hf_status hf_hybrid_forward(const hf_config *cfg, const uint16_t *Q, const uint16_t *Kc,
                            const uint16_t *Vc, int32_t slot_stride,
                            const int32_t *slot_map /* host */, int32_t n_win,
                            const float *S, const float *z, uint16_t *O, int32_t *idx_out,
                            void *ws, void *stream);

/* Key-block pooling for the pooled-key cache (English technical summary,
 * section 2.A.2: the block importance scores use pooled key blocks).  The
 * workspace keeps the pooled keys of every ring slot, fp32 [b, H, W, d/4, bpf, 4]
 * (W = cfg->window_frames slots), between calls; a frame's key blocks do not
 * change while it stays in the window, so they need to be pooled only once,
 * when the frame is written into its slot.  This call pools the key blocks
 * of the ring slots slots[0..n_slots) (host array of distinct slots in
 * [0, W)) of Kc (bf16 [b, H, W, slot_stride, d]) into that cache.  The
 * arithmetic is that of hf_block_scores, so the cached values are identical
 * to the ones hf_hybrid_forward recomputes.  n_slots = 0 is a no-op. */
HF_API hf_status hf_pool_keys(const hf_config *cfg, const uint16_t *Kc, int32_t slot_stride,
                              const int32_t *slots /* host */, int32_t n_slots, void *ws, void *stream);

/* Writes a chunk's keys and values into the K/V ring (the sliding window of
 * English technical summary, section 2.A.2: a new chunk's frames take the
 * slots of the frames it evicts, which must already have been absorbed).
 * K_src, V_src: bf16 [b, H, n_frames, tokens_per_frame, d], contiguous, in
 * device memory or in host memory (pinned host memory lets the copy run
 * asynchronously and overlap other work); Kc, Vc: the ring, bf16
 * [b, H, W, slot_stride, d] in device memory (W = cfg->window_frames slots).
 * Frame f goes to rows [0, tokens_per_frame) of slot slots[f] (host array of
 * n_frames distinct slots in [0, W), 1 <= n_frames <= W).  One pitched copy
 * per frame and tensor (rows = heads), asynchronous on `stream`; the caller
 * keeps the sources alive until the stream reaches this point.  Pooled keys
 * of the written slots are stale afterwards: call hf_pool_keys for them. */
HF_API hf_status hf_ring_write(const hf_config *cfg, const uint16_t *K_src, const uint16_t *V_src,
                               uint16_t *Kc, uint16_t *Vc, int32_t slot_stride,
                               const int32_t *slots /* host */, int32_t n_frames, void *stream);

/* Relative temporal RoPE pre-step (English technical summary, section 2.C
 * "Stability Enhancements": temporal RoPE indices are held under one fixed
 * upper bound in training and inference, positions taken as relative
 * offsets).  Rotary embedding (RoFormer) on channel pairs (2i, 2i+1),
 * i < rot_dims/2: angle p * theta_base^(-2i/rot_dims), where p is the
 * frame's offset inside the current window (offsets[f], host) clamped to
 * [0, max_offset]; channels >= rot_dims are copied unchanged.  src, dst: bf16
 * (device), element (h, f, t, c) at h*head_stride + slots[f]*frame_stride +
 * t*head_dim + c, t < tokens_per_frame (rows between tokens_per_frame and
 * the frame stride are not touched); dst may equal src (in place).  slots:
 * host array of n_frames distinct values in [0, 64).  rot_dims: multiple of
 * 8 in [0, head_dim]; strides: multiples of 8 elements.  Rotate the chunk's
 * queries and the window's keys (from an unrotated ring into a rotated copy,
 * so that no stored value is rotated twice) before the forward; the values
 * and the linear state are not rotated.  Asynchronous on `stream`. */
HF_API hf_status hf_rope_relative(const hf_config *cfg, const uint16_t *src, uint16_t *dst,
                                  int64_t head_stride, int64_t frame_stride,
                                  const int32_t *slots /* host */, const int32_t *offsets /* host */,
                                  int32_t n_frames, int32_t max_offset, int32_t rot_dims,
                                  float theta_base, void *stream);

/* Flags of hf_hybrid_forward_ex. */
#define HF_FWD_CACHED_KEYS 1u  /* take the window's pooled keys from the cache
                                  (every slot of the window pooled by hf_pool_keys,
                                  or by an earlier forward, since it was last written);
                                  only the chunk's queries are pooled */
#define HF_FWD_STATE_PREPARED 2u /* the workspace already holds the state as the
                                  linear read's tensor-core operand: S has not
                                  changed since the last hf_absorb_evicted(_strided)
                                  or forward with this workspace (a fresh, zeroed
                                  workspace holds the operand of S = 0); the forward
                                  then does not read S (may be NULL) */
#define HF_FWD_AFTER_POOL_KEYS 4u /* the last kernel launched on `stream` before
                                  this call is hf_pool_keys, and every kernel that
                                  wrote Q or S finished before that one started:
                                  the forward's first kernel then starts while the
                                  key pooling still runs (programmatic dependent
                                  launch), reading Q and S meanwhile, and waits for
                                  it only before it reads the pooled keys */

/* Number of timing points of hf_hybrid_forward_ex / _profiled. */
#define HF_FWD_EVENTS 4

/* hf_hybrid_forward with options: `flags` (HF_FWD_CACHED_KEYS,
 * HF_FWD_STATE_PREPARED, HF_FWD_AFTER_POOL_KEYS, or 0), per-kernel timing, `events` as in
 * hf_hybrid_forward_profiled (may be NULL), and `state_ready` (a cudaEvent_t,
 * or NULL): the attention kernel, the only one that reads the state (its
 * operand and z), waits for it on `stream`, so the key pooling and the
 * prologue (selection) may run while an absorb on another stream is still
 * producing the state.  Without HF_FWD_CACHED_KEYS every call pools the keys
 * of the whole window (and leaves them in the cache). */
HF_API hf_status hf_hybrid_forward_ex(const hf_config *cfg, const uint16_t *Q, const uint16_t *Kc,
                                      const uint16_t *Vc, int32_t slot_stride,
                                      const int32_t *slot_map /* host */, int32_t n_win,
                                      const float *S, const float *z, uint16_t *O, int32_t *idx_out,
                                      void *ws, void *stream, uint32_t flags,
                                      void *const *events /* host, HF_FWD_EVENTS entries, or NULL */,
                                      void *state_ready /* cudaEvent_t or NULL */);

/* hf_hybrid_forward with per-kernel timing.  The forward runs at most three
 * kernels: the window's key pooling (skipped with HF_FWD_CACHED_KEYS), the
 * prologue (query pooling, the state as the epilogue's tensor-core operand,
 * scores, top-K, the attention kernel's work split) and the attention kernel
 * (sparse softmax attention with the linear read and the sum fused in).
 * events[0..3] (cudaEvent_t handles created by the caller, or NULL for none)
 * are recorded on `stream` before the key pooling, before the prologue,
 * before the attention kernel and after it.  The results are identical to
 * hf_hybrid_forward.  When `stream` is being captured into a CUDA graph the
 * events are captured as external event records, so they time every replay
 * of the graph. */
HF_API hf_status hf_hybrid_forward_profiled(const hf_config *cfg, const uint16_t *Q, const uint16_t *Kc,
                                            const uint16_t *Vc, int32_t slot_stride,
                                            const int32_t *slot_map /* host */, int32_t n_win,
                                            const float *S, const float *z, uint16_t *O,
                                            int32_t *idx_out, void *ws, void *stream,
                                            void *const *events /* host, HF_FWD_EVENTS entries */);

/* Size of the static device scratch that hf_hybrid_forward_noalloc uses in
 * place of a workspace: 16 MiB, enough for the workspace (without its
 * split-pair part, see below) of a 40-head,
 * d = 128 layer with 1560-token frames, a 9-frame window, 3-frame chunks and
 * block 64 (about 9.5 MB). */
#define HF_NOALLOC_SCRATCH_BYTES (16u << 20)

/* The last HF_SPLIT_PARTIAL_BYTES(head_dim) bytes of hf_workspace_size() hold
 * the partial results of tile pairs that the attention kernel cuts between
 * CTAs to balance its work (every CTA takes an equal share of all pairs'
 * rounds, weighted by their MMA work).  A forward without them runs whole
 * pairs per CTA instead: same results up to rounding, less even work.
 * hf_hybrid_forward_noalloc runs that way. */
#define HF_SPLIT_PARTIAL_BYTES(head_dim) (160u * 2u * 2u * 128u * ((unsigned)(head_dim) + 4u) * 4u)

/* hf_hybrid_forward for callers that cannot allocate device memory.  The
 * paper has no counterpart: this is a deployment convenience.
 *
 * Some callers have no way to hand over a workspace: a custom-operator
 * interface that passes only inputs, outputs and a stream; code that runs
 * while a stream is being captured into a CUDA graph, where cudaMalloc is
 * not allowed; an engine that keeps every byte of the device in its own
 * pool.  This entry point takes the same arguments as hf_hybrid_forward
 * except `ws`, and runs the same kernels with the workspace placed in a
 * static device array of HF_NOALLOC_SCRATCH_BYTES that the library defines.
 * The caller still passes (and owns) every input and output.  Nothing is
 * allocated or freed: no cudaMalloc, no cudaFree, no allocating library call.
 *
 *   - Memory: every device that loads the library holds one copy of the
 *     array until the process exits.
 *   - Limit: the scratch stands in for the workspace without its split-pair
 *     part (hf_workspace_size() - HF_SPLIT_PARTIAL_BYTES(head_dim)); a
 *     configuration that needs more than HF_NOALLOC_SCRATCH_BYTES is rejected
 *     with HF_ERR_UNSUPPORTED before anything is launched; use
 *     hf_hybrid_forward for it.
 *   - Set-up: the first call on a device (the calling thread's current
 *     device, which must be the device of `stream` and of the buffers) looks
 *     up the array's device address with cudaGetSymbolAddress, which may load
 *     the library's module on that device.  Make that first call before any
 *     stream capture.  Later calls on the device reuse the address for the
 *     rest of the process.  A cudaDeviceReset (or anything else that destroys
 *     the device's primary context) can move the array: do not call this
 *     entry point on that device after such a reset in the same process.
 *   - Sharing: every call on a device uses the same array, and the array
 *     keeps whatever the last call left in it.  All of it is rewritten before
 *     it is read except the status word, which starts at zero when the
 *     library loads and is cleared by hf_get_device_status.  Two calls whose
 *     kernels may overlap on the GPU (different streams with no ordering
 *     between them) race on the array and give wrong results: order them.
 *   - Device-side errors (a bounded wait that ran out, a bad index) go to
 *     the array's status word.  *status_word (host, may be NULL) receives its
 *     device address; pass that address as `ws` to hf_get_device_status.
 */
HF_API hf_status hf_hybrid_forward_noalloc(const hf_config *cfg, const uint16_t *Q, const uint16_t *Kc,
                                           const uint16_t *Vc, int32_t slot_stride,
                                           const int32_t *slot_map /* host */, int32_t n_win,
                                           const float *S, const float *z, uint16_t *O, int32_t *idx_out,
                                           void **status_word /* host, may be NULL */, void *stream);

/* Synchronises `stream`, reads and clears the workspace status word.
 * Returns HF_OK, HF_ERR_TIMEOUT or HF_ERR_DEVICE_CHECK (the first device-
 * side error since the last call), or HF_ERR_CUDA.  *site (host, may be
 * NULL) receives the code of the wait or check that failed. */
HF_API hf_status hf_get_device_status(void *ws, void *stream, int32_t *site);

/* Diagnostic: launches one tiny kernel that waits on a barrier nothing
 * will ever release, with a limit of `limit_us` microseconds (1..100000),
 * so that the bounded-wait path can be exercised without hanging anything;
 * afterwards hf_get_device_status reports HF_ERR_TIMEOUT. */
HF_API hf_status hf_selftest_wait_timeout(void *ws, int32_t limit_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* HF_H */
