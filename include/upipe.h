/*
 * upipe.h - C ABI of libupipe: the causal GQA attention layer computed one
 * head chunk at a time with one reused workspace, on a single GB300 (sm_103a).
 *
 * The operation.  Untied Ulysses / UPipe ("Untied Ulysses: Memory-Efficient
 * Context Parallelism via Headwise Chunking"; memeeeeeex.com article, section
 * "Untied Ulysses (UPipe)"; talk transcript on liquidgold.cc): the query heads
 * a GPU owns are split into chunks processed one after another; each chunk
 * (re)computes its heads, runs their attention over the whole sequence, and
 * stores its partial result, while the next chunk reuses the buffers the
 * previous one allocated.  On one GPU this is the rank-local work of one
 * Ulysses rank with the all-to-all exchanges left out.  Per chunk c of
 * ``chunk_heads`` query heads h (kv head floor(h / (Hq/Hkv))):
 *     q_h = RoPE(Norm_q(x Wq_h^T)),  k = RoPE(Norm_k(x Wk_g^T)),  v = x Wv_g^T
 *     o_h = softmax(q_h k^T / sqrt(d), causal) v,  lse_h = log-sum-exp of a row
 *     out += sum_{h in c} o_h Wo[:, h*d:(h+1)*d]^T
 * Norm is the per-head RMSNorm of the Qwen3 geometry (qk_norm = 1) and the
 * identity otherwise; RoPE rotates pairs (i, i + d/2) by pos * theta^(-2i/d).
 *
 * Conventions for every call.
 *  - bf16 tensors are passed as upipe_bf16 (raw 16-bit storage); all matrices
 *    are row-major with the nn.Linear weight layout [out_features, in_features]:
 *      x, dout [S, hidden];  Wq [Hq*d, hidden];  Wk, Wv [Hkv*d, hidden];
 *      Wo [hidden, Hq*d];    q_norm_w, k_norm_w [d] (fp32; NULL means ones).
 *  - Pointers named x, W*, out, lse, d*, workspace are DEVICE pointers of the
 *    current CUDA device; every buffer must be 16-byte aligned.
 *  - ``stream`` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    enqueue work and return; nothing is synchronised.  With more than one
 *    chunk, upipe_attn_fwd forks part of its work onto a library-owned
 *    high-priority stream of the device (created by the first such call) and
 *    joins it back with events before it returns, so its work is ordered like
 *    one launch sequence on ``stream``.  Two calls in flight at once must not
 *    share a workspace.
 *  - Ownership: the caller owns every buffer.  The library allocates no device
 *    or host memory of its own: upipe_attn_fwd creates only the one stream per
 *    device named above and three events per call, upipe_offload /
 *    upipe_prefetch one copy stream per device and two events per copy (one
 *    released by upipe_copy_join); all temporaries live in ``workspace``.
 *  - Errors: every argument is validated on the host before the first launch;
 *    a failed check returns a code and launches nothing.  A device-side wait
 *    that exceeds its time limit, or a projected value outside the fp16 range,
 *    is reported by upipe_last_error().
 *  - Precision: inputs are bf16 and every contraction accumulates in fp32.
 *    The per-chunk q, k, v (after norm and RoPE) and the attention kernels'
 *    probabilities and gradients are held in fp16, whose 11 significant bits
 *    (bf16: 8) keep the layer within max 2e-2 / mean 2e-3 (relative to unit
 *    scale) and |lse| 1e-3 of the float64 definition; q, k and v must
 *    therefore lie within fp16's range (|v| <= 65504, else UPIPE_ERR_RANGE).
 *    The backward scales dO and dS by exact powers of two derived on the
 *    device from norms of dout, Wo, v and dO, so gradients of any magnitude
 *    keep their precision.  The attention output o (attn_o) is bf16 and out,
 *    lse and all gradients are fp32.
 */
#ifndef UPIPE_H_
#define UPIPE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t upipe_bf16;

/* Geometry of one attention layer and its head chunking.
 *   S            tokens (full sequence), 1 <= S <= 2^31 - 256
 *   hidden       model width, a multiple of 128
 *   Hq, Hkv      query and key/value heads; Hkv divides Hq
 *   d            head dimension: 64 or 128
 *   chunk_heads  query heads per chunk; divides Hq, and either
 *                (Hq/Hkv) divides chunk_heads or chunk_heads divides (Hq/Hkv)
 *   rope_theta   RoPE base (> 0)
 *   qk_norm      0: no q/k normalisation (Llama); 1: per-head RMSNorm on q and
 *                k before RoPE (Qwen3)
 *   norm_eps     RMSNorm epsilon (added to mean(v^2) inside the root) */
typedef struct {
  int64_t S;
  int32_t hidden, Hq, Hkv, d, chunk_heads;
  double rope_theta;
  int32_t qk_norm;
  float norm_eps;
} upipe_shape_t;

enum {
  UPIPE_OK = 0,
  UPIPE_ERR_INVALID_ARG = 1,          /* NULL pointer, bad size, misalignment */
  UPIPE_ERR_UNSUPPORTED = 2,          /* a shape the library does not handle */
  UPIPE_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes < upipe_workspace_bytes()  */
  UPIPE_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed    */
  UPIPE_ERR_DEVICE_TIMEOUT = 5,       /* a kernel's bounded wait expired      */
  UPIPE_ERR_RANGE = 6,                /* a projected q, k or v value exceeds
                                         the fp16 range (|v| > 65504)        */
  UPIPE_ERR_BOUNDS = 7,               /* debug builds only: a device-side
                                         bounds check of a global access
                                         failed (the access was skipped)     */
  UPIPE_ERR_TARGET = 8                /* a loss target id outside
                                         [0, vocab) (its row's loss is NaN)  */
};

/* Workspace bytes needed by upipe_attn_fwd (mode 0) or upipe_attn_bwd
 * (mode 1) for this shape, or 0 if the shape is invalid.  Pure host function.
 * Mode 2 is mode 0 plus a third chunk buffer (S * chunk_heads * d bf16): given
 * that much, upipe_attn_fwd adds two chunks' partial results into out per
 * pass (see there).  Mode 3 is upipe_attn_fwd_fused's: mode 0 without the
 * second chunk buffer (S * chunk_heads * d bf16 less).
 * The bytes are affine in chunk_heads: the per-chunk Q/O (and backward) parts
 * scale with chunk_heads, the K/V part is one KV group (or chunk_heads/(Hq/Hkv)
 * groups when a chunk spans several), plus RoPE tables of
 * ((S >> 10) + 1 + 2 * 1024) * d/2 float2 entries.  Every chunk runs in these same
 * buffers, which is how UPipe saves memory (memeeeeeex.com, "Untied Ulysses
 * (UPipe)": the chunks reuse one set of buffers). */
size_t upipe_workspace_bytes(const upipe_shape_t* shape, int mode);

/* Forward of the layer, chunk by chunk (the UPipe loop).
 *   out   [S, hidden] fp32, overwritten (the first chunk stores, later chunks
 *         add their Wo-slice partial results)
 *   lse   [Hq, S] fp32 natural-log log-sum-exp of each head's scaled scores
 *   attn_o  NULL, or [S, Hq*d] bf16: receives every head's attention output
 *         o_h at columns h*d.  Keep it for upipe_attn_bwd_saved_o (the
 *         backward then skips recomputing the attention forward), or use it
 *         to check that o_h does not depend on chunk_heads.
 *   workspace / ws_bytes: device buffer of at least
 *         upipe_workspace_bytes(shape, 0) bytes, 256-byte aligned
 * Paired accumulates: with three or more chunks, when the forward forks and
 * either attn_o is given or ws_bytes >= upipe_workspace_bytes(shape, 2), each
 * Wo-slice accumulate adds two chunks (K = 2 * chunk_heads * d) and out is
 * read and written half as often.  out then differs from the unpaired
 * forward by the order of its fp32 additions (~1e-7 relative); lse and the
 * attention output are bit-identical.
 * Returns UPIPE_OK or an error code (nothing launched on error). */
int upipe_attn_fwd(const upipe_shape_t* shape, const upipe_bf16* x, const upipe_bf16* Wq,
                   const upipe_bf16* Wk, const upipe_bf16* Wv, const upipe_bf16* Wo,
                   const float* q_norm_w, const float* k_norm_w, float* out, float* lse,
                   void* workspace, size_t ws_bytes, upipe_bf16* attn_o, void* stream);

/* Forward of the layer with each chunk's partial result added into out by the
 * attention kernel itself (memeeeeeex.com, "Untied Ulysses (UPipe)": each
 * chunk stores its partial result; here without an attention-output buffer).
 * Same arguments and results as upipe_attn_fwd without attn_o:
 *   out   [S, hidden] fp32, overwritten: zeroed on ``stream``, then every
 *         head's o_h Wo[:, h*d:(h+1)*d]^T is added by the CTAs that computed
 *         o_h (fp32 adds in L2, in no fixed order: out matches
 *         upipe_attn_fwd's to fp32 rounding, ~1e-6 relative, and may differ
 *         in its last bits between runs)
 *   lse   [Hq, S] fp32, bit-identical to upipe_attn_fwd's
 *   workspace / ws_bytes: at least upipe_workspace_bytes(shape, 3) bytes,
 *         256-byte aligned (no O buffer: one chunk's Q, the K/V of its group
 *         and the RoPE tables)
 * Every launch runs on ``stream`` (no side stream, no events).
 * Returns UPIPE_OK or an error code (nothing launched on error). */
int upipe_attn_fwd_fused(const upipe_shape_t* shape, const upipe_bf16* x, const upipe_bf16* Wq,
                         const upipe_bf16* Wk, const upipe_bf16* Wv, const upipe_bf16* Wo,
                         const float* q_norm_w, const float* k_norm_w, float* out, float* lse,
                         void* workspace, size_t ws_bytes, void* stream);

/* Backward of the layer for L = sum(out * dout), chunk by chunk, recomputing
 * each chunk's Q/K/V and attention output in the reused workspace (activation
 * recomputation: aipmzone.com / dimanyen.com, "activation checkpointing").
 *   dout  [S, hidden] bf16 upstream gradient
 *   lse   [Hq, S] fp32 from upipe_attn_fwd on the same inputs
 *   dx    [S, hidden] fp32, overwritten
 *   dWq [Hq*d, hidden], dWk/dWv [Hkv*d, hidden], dWo [hidden, Hq*d]: fp32,
 *         overwritten
 *   dq_norm_w, dk_norm_w [d] fp32, overwritten when qk_norm = 1 (may be NULL
 *         when qk_norm = 0)
 *   workspace: at least upipe_workspace_bytes(shape, 1) bytes. */
int upipe_attn_bwd(const upipe_shape_t* shape, const upipe_bf16* x, const upipe_bf16* Wq,
                   const upipe_bf16* Wk, const upipe_bf16* Wv, const upipe_bf16* Wo,
                   const float* q_norm_w, const float* k_norm_w, const upipe_bf16* dout,
                   const float* lse, float* dx, float* dWq, float* dWk, float* dWv, float* dWo,
                   float* dq_norm_w, float* dk_norm_w, void* workspace, size_t ws_bytes,
                   void* stream);

/* The same backward, with the attention output saved by the forward instead
 * of recomputed.  upipe_attn_bwd recomputes every chunk's attention forward
 * (4*d FLOPs per causal pair and head, about 30% of the backward's work) so
 * that only the chunk-sized workspace holds activations; a caller that can
 * keep the full attention output of the layer (S * Hq * d bf16, e.g. 1 GiB for
 * 4 heads of d = 128 over 1M tokens) passes it here and saves that work.
 * This is the memory / throughput trade of the chunk-size choice
 * (memeeeeeex.com "Results": larger chunks use more memory and run slightly
 * faster), taken one step further.
 *   attn_o  [S, Hq*d] bf16, as written by upipe_attn_fwd(..., attn_o, ...) on
 *           the same inputs (required: NULL is UPIPE_ERR_INVALID_ARG)
 * Every other argument, the workspace size and the results are those of
 * upipe_attn_bwd. */
int upipe_attn_bwd_saved_o(const upipe_shape_t* shape, const upipe_bf16* x, const upipe_bf16* Wq,
                           const upipe_bf16* Wk, const upipe_bf16* Wv, const upipe_bf16* Wo,
                           const float* q_norm_w, const float* k_norm_w, const upipe_bf16* dout,
                           const float* lse, const upipe_bf16* attn_o, float* dx, float* dWq,
                           float* dWk, float* dWv, float* dWo, float* dq_norm_w,
                           float* dk_norm_w, void* workspace, size_t ws_bytes, void* stream);

/* Forward for callers that cannot allocate device memory: code running where
 * cudaMalloc is not allowed or not wanted (inside a graph-building or
 * real-time section, under an external allocator that forbids extra device
 * allocations, or in a plugin that only receives its inputs' and outputs'
 * pointers).  The paper has no counterpart; this is a convenience of the
 * library.  Same arguments and results as upipe_attn_fwd minus the workspace
 * and attn_o: the workspace is a static device array of
 * UPIPE_STATIC_SCRATCH_BYTES (64 MiB) compiled into the library, which every
 * GPU that loads the library holds until the process exits.
 *  - Shapes whose upipe_workspace_bytes(shape, 0) exceeds
 *    UPIPE_STATIC_SCRATCH_BYTES are rejected with
 *    UPIPE_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 *  - The first call on each device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Allocates nothing: no cudaMalloc/cudaFree or allocating library call.
 *    Unlike upipe_attn_fwd it keeps every launch on ``stream``: it uses no
 *    side stream and creates no events.
 *  - Every call shares the one array and leaves its contents behind; nothing
 *    in it needs to start at zero.  Calls that overlap on the GPU (different
 *    streams, or host threads racing) race on the array: serialise them. */
#define UPIPE_STATIC_SCRATCH_BYTES (64u << 20)
int upipe_attn_fwd_noalloc(const upipe_shape_t* shape, const upipe_bf16* x, const upipe_bf16* Wq,
                           const upipe_bf16* Wk, const upipe_bf16* Wv, const upipe_bf16* Wo,
                           const float* q_norm_w, const float* k_norm_w, float* out, float* lse,
                           void* stream);

/* Measurement hook (no counterpart on the pages; used by the benchmark to
 * time one kernel live inside a layer call).  While attached, each launch of
 * the selected kernel made by upipe_attn_fwd / upipe_attn_bwd records
 * start_events[i] just before and end_events[i] just after itself on the
 * call's stream, for i = 0, 1, ... < capacity; later launches are not timed.
 *   kernel 0: the attention forward kernel;  kernel 1: the attention backward
 *   kernel 2: the Wo-slice accumulate GEMMs that run on the call's stream
 *             with every SM (the last chunk's, or the last pair's when the
 *             accumulates are paired; every chunk's when the forward does not
 *             fork), not those beside the next attention
 *   kernel 3: the RoPE/RMSNorm backward of dQ (one per chunk) and of dK
 *             (one per KV group), in launch order
 *   kernel 4: the fp32 -> bf16 hi/lo split of dV (one per KV group)
 *   kernel 5: the attention forward kernel of upipe_attn_fwd_fused (with its
 *             fused Wo-slice accumulate)
 *   start_events/end_events: caller-created cudaEvent_t handles (timing
 *   enabled), owned by the caller.  capacity 0 detaches.
 * upipe_profile_count() returns how many launches were recorded since the
 * last attach.  Host-side state shared by all threads: not thread-safe. */
void upipe_profile_attach(int kernel, void* const* start_events, void* const* end_events,
                          int capacity);
int upipe_profile_count(void);

/* Failure-detection self-test (no counterpart on the pages).  Enqueues a
 * one-CTA kernel whose device-side waits can never be satisfied and expire
 * after limit_us microseconds (1 .. 1e6), exactly as a stuck wait inside the
 * layer kernels would: the kernel records UPIPE_ERR_DEVICE_TIMEOUT in the
 * device error word and returns, without faulting.  The next
 * upipe_last_error() reports it; the context stays usable.
 * Returns UPIPE_OK once enqueued, UPIPE_ERR_INVALID_ARG for a bad limit. */
int upipe_selftest_wait_timeout(int limit_us, void* stream);

/* ------------------------------------------------------------------------
 * The sequence-tiled MLP of the decoder layer (no counterpart in the chunked
 * attention itself).  The pages' memory stack tiles the element-wise parts of
 * the layer, the MLPs and the loss, along the sequence so that no buffer as
 * long as the sequence is created (memeeeeeex.com article, the stack section
 * on Arctic sequence-length training; liquidgold.cc talk transcript).  The MLP
 * is the bias-free SwiGLU MLP of the Llama / Qwen3 models:
 *     y = (silu(x Wg^T) * (x Wu^T)) Wd^T,   silu(v) = v / (1 + e^-v)
 * computed over tiles of tile_rows tokens; the [tile_rows, ffn]
 * intermediates live in the workspace and are reused by every tile.  A
 * token's output depends on that token alone, so tiling changes memory, not
 * the result.
 *   S          tokens, 1 <= S <= 2^31 - 256
 *   hidden     model width, a multiple of 128
 *   ffn        MLP width, a multiple of 128
 *   tile_rows  tokens per tile, a multiple of 128 (S itself when shorter)
 * Layouts (row-major, nn.Linear weights): x, dy [S, hidden] bf16;
 * Wg, Wu [ffn, hidden] bf16; Wd [hidden, ffn] bf16; y, dx [S, hidden] fp32;
 * dWg, dWu [ffn, hidden] fp32; dWd [hidden, ffn] fp32.  The per-tile
 * intermediates a, dg, du are held in bf16, every contraction accumulates in
 * fp32.  Device pointers, 16-byte aligned; the workspace 256-byte aligned.
 * ------------------------------------------------------------------------ */
typedef struct {
  int64_t S;
  int32_t hidden, ffn, tile_rows;
} upipe_mlp_shape_t;

/* Workspace bytes of upipe_mlp_fwd (mode 0: a, min(tile_rows, S) x ffn bf16)
 * or upipe_mlp_bwd (mode 1: a, dg, du bf16 and dA fp32 of one tile), or 0 for
 * an invalid shape or mode.  Pure host function. */
size_t upipe_mlp_workspace_bytes(const upipe_mlp_shape_t* shape, int mode);

/* y = MLP(x), tile by tile.  y is overwritten (every row is stored once).
 * Returns UPIPE_OK or an error code (nothing launched on error). */
int upipe_mlp_fwd(const upipe_mlp_shape_t* shape, const upipe_bf16* x, const upipe_bf16* Wg,
                  const upipe_bf16* Wu, const upipe_bf16* Wd, float* y, void* workspace,
                  size_t ws_bytes, void* stream);

/* Gradients of L = sum(y * dy): dx (overwritten, row by row), dWg, dWu, dWd
 * (zeroed, then accumulated over the tiles with fp32 reduce-adds in no fixed
 * order).  Each tile recomputes its gate and up projections.
 * Returns UPIPE_OK or an error code (nothing launched on error). */
int upipe_mlp_bwd(const upipe_mlp_shape_t* shape, const upipe_bf16* x, const upipe_bf16* Wg,
                  const upipe_bf16* Wu, const upipe_bf16* Wd, const upipe_bf16* dy, float* dx,
                  float* dWg, float* dWu, float* dWd, void* workspace, size_t ws_bytes,
                  void* stream);

/* ------------------------------------------------------------------------
 * The sequence-tiled cross-entropy loss of the model's last layer (the
 * pages' stack tiles the loss along the sequence, as it does the MLPs:
 * memeeeeeex.com article, the stack section on Arctic sequence-length
 * training).  With logits z = h W^T over a vocabulary of V words,
 *     lse_i = log sum_v exp(z_iv),   loss_i = lse_i - z_i[t_i]
 * computed over tiles of tile_rows tokens: the [tile_rows, V] logits are
 * never stored in the forward (the logits GEMM's epilogue reduces them to
 * per-row partials); the backward recomputes them per tile.
 *   S, hidden, tile_rows as for the MLP; vocab a multiple of 128
 * Layouts: h [S, hidden] bf16; W [vocab, hidden] bf16 (nn.Linear);
 * targets [S] int32 in [0, vocab); loss_rows, lse [S] fp32 (natural log);
 * dh [S, hidden] fp32; dW [vocab, hidden] fp32.  dz is held in bf16 per
 * tile; every contraction accumulates in fp32.
 * ------------------------------------------------------------------------ */
typedef struct {
  int64_t S;
  int32_t hidden, vocab, tile_rows;
} upipe_loss_shape_t;

/* Workspace bytes of upipe_loss_fwd (mode 0: one tile's per-row partials,
 * tile x vocab/256 (or /128) float2, and target logits) or upipe_loss_bwd
 * (mode 1: one tile's dz, tile x vocab bf16), or 0 for an invalid shape or
 * mode.  Pure host function. */
size_t upipe_loss_workspace_bytes(const upipe_loss_shape_t* shape, int mode);

/* Per-token losses and log-sum-exps, tile by tile (both overwritten).  A
 * target outside [0, vocab) gives its row a NaN loss and UPIPE_ERR_TARGET
 * through upipe_last_error().
 * Returns UPIPE_OK or an error code (nothing launched on error). */
int upipe_loss_fwd(const upipe_loss_shape_t* shape, const upipe_bf16* h, const upipe_bf16* W,
                   const int32_t* targets, float* loss_rows, float* lse, void* workspace,
                   size_t ws_bytes, void* stream);

/* Gradients of L = scale * sum_i loss_i (scale = 1/S for the mean) given the
 * forward's lse: dh (overwritten, row by row) and dW (zeroed, then
 * accumulated over the tiles with fp32 reduce-adds in no fixed order).
 * Returns UPIPE_OK or an error code (nothing launched on error). */
int upipe_loss_bwd(const upipe_loss_shape_t* shape, const upipe_bf16* h, const upipe_bf16* W,
                   const int32_t* targets, const float* lse, float scale, float* dh, float* dW,
                   void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Offload of block inputs to host memory and their prefetch back (the pages'
 * CPU-offload step: a transformer block's input leaves the GPU while it is
 * not needed and is prefetched before the backward reaches that block, the
 * copies running under compute; memeeeeeex.com article, the stack section on
 * CPU offload).  Each call enqueues one asynchronous copy on a library-owned
 * copy stream of the current device (created by the first call), ordered
 * after everything enqueued on ``stream`` so far, and returns a ticket;
 * upipe_copy_join(ticket, consumer_stream) makes the consumer's stream wait
 * for the copy and releases the ticket (every ticket must be joined once).
 *   dev_src / dev_dst   device memory of the current device
 *   host_dst / host_src page-locked host memory (cudaHostAlloc or
 *                       cudaHostRegister; pageable memory is refused: its
 *                       copies would not run asynchronously)
 *   bytes               > 0
 * The caller must not touch the source or destination until the copy is
 * joined.  Returns UPIPE_OK, UPIPE_ERR_INVALID_ARG (a NULL pointer, zero
 * bytes, or memory of the wrong kind; nothing enqueued) or UPIPE_ERR_CUDA.
 * ------------------------------------------------------------------------ */
int upipe_offload(const void* dev_src, void* host_dst, size_t bytes, void* stream, void** ticket);
int upipe_prefetch(const void* host_src, void* dev_dst, size_t bytes, void* stream,
                   void** ticket);
int upipe_copy_join(void* ticket, void* stream);

/* 1 if this library was built with device-side bounds checks (the debug
 * build: UPIPE_DEBUG_BOUNDS), else 0.  In that build every plain (non-TMA)
 * global load and store of the kernels is checked against the extent of its
 * view as the launch declares it; a failed check skips the access and
 * records UPIPE_ERR_BOUNDS for upipe_last_error().  It stands in for a
 * memory checker (no such checker runs on the GPUs this library is tested
 * on).  Host function. */
int upipe_debug_bounds(void);

/* Bounds-check self-test (no counterpart on the pages).  Runs a one-thread
 * kernel that asks to write one element past a declared view (the element
 * lies inside the underlying array, so the write is harmless either way) and
 * waits for it on ``stream``.  *written receives 1 if the write happened.
 * Debug build: the check refuses it (*written = 0) and the next
 * upipe_last_error() returns UPIPE_ERR_BOUNDS.  Release build: the write
 * happens (*written = 1) and nothing is reported.
 * Returns UPIPE_OK, UPIPE_ERR_INVALID_ARG (written NULL) or UPIPE_ERR_CUDA. */
int upipe_selftest_bounds(void* stream, int* written);

/* The output-tile walk of the library's persistent GEMM (no counterpart on
 * the pages): the host copy of the device function by which every GEMM
 * launch maps a tile index to its work.  A launch covers num_m 128-row
 * blocks x num_n column tiles x ksplit partitions of the kb_total 64-wide K
 * blocks; each CTA takes tile indices blockIdx.x, blockIdx.x + gridDim.x, ...
 * For tile t the call writes out[4t .. 4t+3] = (row block, column tile,
 * first K block, one past the last K block); the K range is empty when the
 * partitions outnumber what kb_total fills.  m_fastest orders the tiles of a
 * partition: 0 column tiles fastest, 1 row blocks fastest, G > 1 row blocks
 * fastest within groups of G row blocks, group after group.  out holds
 * out_len int32 elements (caller-owned host memory, at least
 * 4 * num_m * num_n * ksplit).  Host function, no device work.
 * Returns UPIPE_OK, or UPIPE_ERR_INVALID_ARG for a count below 1, a negative
 * m_fastest, more than 2^31 - 1 tiles, m_fastest * num_n above 2^31 - 1, or
 * out NULL or short. */
int upipe_gemm_tile_order(int num_m, int num_n, int kb_total, int ksplit, int m_fastest,
                          int32_t* out, int64_t out_len);

/* Synchronises the current device, then returns and clears the device error
 * word (UPIPE_OK, UPIPE_ERR_DEVICE_TIMEOUT, UPIPE_ERR_RANGE, UPIPE_ERR_TARGET
 * or, in the debug build, UPIPE_ERR_BOUNDS: the first error a kernel recorded
 * since the last call), or UPIPE_ERR_CUDA if the device reports a CUDA
 * error. */
int upipe_last_error(void);

/* Static description of an error code. */
const char* upipe_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* UPIPE_H_ */
