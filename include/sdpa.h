/*
 * sdpa.h — C ABI of the GB300 (sm_103a) fused scaled-dot-product attention
 * library for training: a flash-style forward that stashes the per-row
 * log-sum-exp, and the matching backward that recomputes the probabilities
 * from it.
 *
 * The operation is scaled dot-product attention as named in the
 * "Scaled_dot_product_attention" thread (discuss.pytorch.org):
 *     out = dropout(softmax(scale * Q K^T + causal)) V
 * with the argument lists of sdpfa_fwd / sdpfa_bwd in test_sdpa_loop_split
 * ("DID loop split for SDPA", NVIDIA/Fuser PR 3711), the E = Ev restriction
 * of the SdpaFwdOp plan (NVIDIA/Fuser issue 2278, "Note to self: next PRs"),
 * and dropout regenerated from (seed, offset) and the absolute element index
 * ("REDO of dropout support for mem eff #102038", pytorch PR 103704, Summary).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are described by sdpa_tensor: a device pointer to bfloat16 data,
 *   the LOGICAL shape [B, H, S, D] and the stride of each logical dim in
 *   ELEMENTS. Any dense order of B, H, S works as long as D is innermost
 *   (stride[3] == 1); BHSE (stride order 3,2,1,0) and BSHE (3,1,2,0) are the
 *   two layouts of test_sdpa_loop_split. Strides of dims of size > 1 must be
 *   multiples of 8 elements (16 bytes) and every base pointer 16-byte aligned.
 * - D (= E = Ev, the head dim of q, k and v) must be a multiple of 8 from 8
 *   to 256. The kernels are built for 64, 128 and 256 (the backward for 128
 *   and 256); a smaller D runs the next larger one, the missing columns being
 *   read as zeros by the TMA loads and never stored, so the results are those
 *   of D itself. An attention bias (sdpa_options.attn_bias) is served up to
 *   D = 128.
 * - Causal masking is top-left aligned: key j is visible to query i iff j <= i.
 * - Ownership: the caller allocates every input, output and workspace; the
 *   library allocates no device memory and keeps no per-call state. Work is
 *   enqueued on `stream` (0 = legacy default stream) and the call returns
 *   without synchronising. Inputs must stay valid until the stream reaches
 *   the work.
 * - Errors: argument problems are reported synchronously and nothing is
 *   launched. SDPA_ERR_CUDA means a launch failed (the CUDA error is
 *   retrievable with cudaGetLastError). Every wait inside the kernels is
 *   bounded; a kernel whose wait runs out records it in a device error word,
 *   which sdpa_check_device() reads (and the entry points read themselves
 *   when the environment variable SDPA_DEBUG_SYNC=1 is set).
 * - Empty problems (B*H*Sq == 0) succeed without launching anything, except
 *   that the backward still zero-fills dk and dv when Sq == 0.
 */
#ifndef SDPA_GB300_H
#define SDPA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream (binary-compatible with cudaStream_t). */
typedef struct CUstream_st* sdpa_stream_t;

typedef struct {
  void* data;          /* device pointer, bfloat16 elements */
  int64_t size[4];     /* logical [B, H, S, D] */
  int64_t stride[4];   /* element strides of the logical dims */
} sdpa_tensor;

typedef enum {
  SDPA_OK = 0,
  SDPA_ERR_INVALID_ARG = 1,    /* shape mismatch, null pointer, p outside [0,1), bad scale */
  SDPA_ERR_UNSUPPORTED = 2,    /* D not a multiple of 8 in [8, 256], D not innermost, an
                                  attention bias with D > 128 or a packed batch, or
                                  B*H*ceil(max(Sq, Sk)/128) above 2^31-1 (launch grids) */
  SDPA_ERR_ALIGNMENT = 3,      /* base or stride not 16-byte aligned */
  SDPA_ERR_CUDA = 4,           /* a CUDA launch or driver call failed */
  SDPA_ERR_DEVICE_TIMEOUT = 5, /* a kernel gave up on a bounded wait */
  SDPA_ERR_WORKSPACE = 6       /* workspace missing or smaller than required */
} sdpa_status;

/*
 * sdpa_fwd — forward of fused attention for training (sdpfa_fwd of
 * test_sdpa_loop_split, "DID loop split for SDPA"; the stashed log-sum-exp
 * of issue "SdpaOpFwd / SdpaOpBwd nodes", NVIDIA/Fuser 2278).
 *   q [B,H,Sq,D], k [B,H,Sk,D], v [B,H,Sk,D]: inputs (read only).
 *   dropout_p in [0,1): probability of dropping an attention weight;
 *     kept weights are scaled by 1/(1-p).
 *   is_causal: nonzero for the top-left causal mask.
 *   scale: softmax scale (> 0, finite); the usual choice is 1/sqrt(D).
 *   seed, offset: Philox4x32-10 key and counter offset of the dropout mask
 *     (ignored when dropout_p == 0). Pass the same values to sdpa_bwd.
 *   out [B,H,Sq,D]: bfloat16 output, any layout allowed for q.
 *   lse: float32 [B,H,Sq], contiguous: natural-log log-sum-exp of each
 *     scaled, masked score row (before dropout).
 * Requires Sk >= 1 whenever B*H*Sq > 0.
 */
sdpa_status sdpa_fwd(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                     double dropout_p, int is_causal, float scale, uint64_t seed,
                     uint64_t offset, sdpa_tensor* out, float* lse, sdpa_stream_t stream);

/*
 * sdpa_bwd_workspace_size — bytes of device workspace sdpa_bwd needs for
 * this problem size: an fp32 dQ accumulator of Dk-wide rows (Dk = 64 for
 * D <= 64, 128 for D <= 128, whose backward runs on 128-wide tiles, and 256
 * above) and two fp32 row vectors, with Sq rounded up to a multiple of 128:
 * B*H*ceil128(Sq)*(Dk + 2)*4 bytes.
 * Returns 0 for an empty problem, and SIZE_MAX when the size does not fit in
 * 62 bits (no workspace then satisfies sdpa_bwd, which returns
 * SDPA_ERR_WORKSPACE).
 */
size_t sdpa_bwd_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t D);

/*
 * sdpa_bwd — backward of fused attention (sdpfa_bwd of test_sdpa_loop_split,
 * "DID loop split for SDPA"): recomputes the probabilities from lse,
 * regenerates the dropout mask from (seed, offset), and writes
 *   dq = scale * dS K,  dk = scale * dS^T Q,  dv = P~^T dout,
 * with dS = P * (dout V^T * keep/(1-p) - rowsum(dout * out)).
 *   dout, q, k, v, out: bfloat16 tensors as in sdpa_fwd (out and lse must be
 *     the forward's results for the same q, k, v, p, is_causal, seed, offset, scale).
 *   lse: float32 [B,H,Sq] contiguous, from sdpa_fwd.
 *   dq [B,H,Sq,D], dk, dv [B,H,Sk,D]: bfloat16 outputs (any allowed layout).
 *   workspace: device memory of at least sdpa_bwd_workspace_size() bytes,
 *     256-byte aligned; its contents on entry do not matter and are
 *     overwritten. It must not be shared by calls in flight at the same time.
 * Launches three kernels on `stream`: preprocess, main, dQ conversion.
 */
sdpa_status sdpa_bwd(const sdpa_tensor* dout, const sdpa_tensor* q, const sdpa_tensor* k,
                     const sdpa_tensor* v, const sdpa_tensor* out, const float* lse,
                     double dropout_p, int is_causal, uint64_t seed, uint64_t offset,
                     float scale, sdpa_tensor* dq, sdpa_tensor* dk, sdpa_tensor* dv,
                     void* workspace, size_t workspace_bytes, sdpa_stream_t stream);

/* Size of the scratch array built into the library for sdpa_bwd_noalloc. */
#define SDPA_BWD_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * sdpa_bwd_noalloc — the same backward as sdpa_bwd, for callers that cannot
 * allocate device memory: code that a host framework hands only its input
 * and output buffers, under rules that forbid private cudaMalloc calls
 * (they would bypass the framework's memory pool and accounting), and
 * latency-critical loops where an allocation, which may synchronise the
 * device, is not acceptable. The pages have no counterpart; this is a
 * convenience of this library.
 *   Arguments are those of sdpa_bwd without the workspace; the caller still
 *   passes every input and output. The workspace comes from one fixed array
 *   of SDPA_BWD_NOALLOC_SCRATCH_BYTES (64 MiB) compiled into the library:
 *   every GPU that loads the library holds it until the process exits.
 *   Problems whose sdpa_bwd_workspace_size() exceeds that maximum are
 *   rejected with SDPA_ERR_WORKSPACE and nothing is launched.
 *   Nothing is allocated: no cudaMalloc or cudaFree, no allocating library
 *   routine. The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.
 *   All calls share the one array, which keeps whatever the last call left
 *   in it (every call overwrites what it reads, so results do not depend on
 *   it). Calls whose work overlaps on the GPU -- e.g. issued to two streams
 *   without ordering between them -- race on the array and give wrong
 *   results; order them on one stream.
 */
sdpa_status sdpa_bwd_noalloc(const sdpa_tensor* dout, const sdpa_tensor* q, const sdpa_tensor* k,
                             const sdpa_tensor* v, const sdpa_tensor* out, const float* lse,
                             double dropout_p, int is_causal, uint64_t seed, uint64_t offset,
                             float scale, sdpa_tensor* dq, sdpa_tensor* dk, sdpa_tensor* dv,
                             sdpa_stream_t stream);

/*
 * sdpa_dropout_mask_debug — writes the keep mask (1 = kept, 0 = dropped) of
 * every element of a [B,H,Sq,Sk] attention problem into `mask` (uint8, device,
 * contiguous [B,H,Sq,Sk]), computed by the same device Philox routine the
 * forward and backward kernels use ("REDO of dropout support for mem eff
 * #102038", Summary: absolute-index RNG). For tests and debugging.
 */
sdpa_status sdpa_dropout_mask_debug(int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                                    double dropout_p, uint64_t seed, uint64_t offset,
                                    uint8_t* mask, sdpa_stream_t stream);

/*
 * sdpa_options — extensions of the forward and backward calls (the *_ex entry
 * points below). A zero-initialised struct, or a NULL pointer, gives exactly
 * the behaviour of sdpa_fwd / sdpa_bwd / sdpa_dropout_mask_debug.
 *
 *   rng_state: NULL, or a device pointer (8-byte aligned) to two uint64
 *     values {seed, offset} that the kernels read when they run, in place of
 *     the seed and offset arguments. The rng state then travels from forward
 *     to backward through device memory, so a captured CUDA graph can be
 *     replayed with a new state written into that buffer between replays
 *     (the graph-safe rng passing of "REDO of dropout support for mem eff
 *     #102038", pytorch PR 103704, Summary). The buffer must hold the same
 *     values when the backward runs as when the forward ran.
 *   batch_offset, head_offset, total_heads: where this call's [B, H] block
 *     sits in a larger problem that is split by batch and head across calls
 *     or devices (the head split of test_sdpa_loop_split, "DID loop split for
 *     SDPA", NVIDIA/Fuser PR 3711). The dropout counter uses the global
 *     batch index batch_offset + b and head index head_offset + h out of
 *     total_heads heads per batch, so each part draws exactly its slice of
 *     the unsplit problem's mask. total_heads = 0 means H (no head split);
 *     otherwise head_offset + H <= total_heads. Offsets must be >= 0.
 *   attn_bias: NULL, or an additive bias B_ij of the attention scores, for
 *     example a relative-position bias (the forum thread's self-attention
 *     with relative positional encoding; attn_bias in the memory-efficient
 *     kernel, PR 103704's priority-order discussion). It is read as torch's
 *     float attn_mask: softmax(scale * Q K^T + B + causal), and lse is that
 *     of the biased scores. bfloat16, logical [B or 1, H or 1, Sq, Sk] (a
 *     size-1 dim, or a stride-0 dim, is shared by every batch / head), keys
 *     contiguous (stride[3] == 1), other strides multiples of 8 elements and
 *     the base 16-byte aligned. Pass the same bias to sdpa_bwd_ex.
 *   dbias: sdpa_bwd_ex only. NULL, or a bfloat16 [B, H, Sq, Sk] tensor
 *     (keys contiguous, aligned as attn_bias) that receives dB = dS, the gradient of the loss with
 *     respect to the biased scores, for every (b, h); positions hidden by
 *     the causal mask get 0. Summing it over a shared dim gives the gradient
 *     of a shared bias. Requires attn_bias.
 *   deterministic: sdpa_bwd_ex only. Nonzero: every 128-key tile stores its
 *     fp32 dQ partials into its own workspace slice and a final kernel adds
 *     them in key-tile order, so dq is bitwise reproducible run to run (the
 *     default reduce-adds partials into one accumulator in whatever order
 *     the tiles finish). It needs the larger workspace that
 *     sdpa_bwd_workspace_size_ex() reports and moves about twice the partials'
 *     bytes through HBM.
 *   dropout_bits, dropout_bits_bytes: NULL, or a device buffer (4-byte
 *     aligned, at least sdpa_dropout_bits_size(B, H, Sq, Sk) bytes) that
 *     carries the dropout keep mask from the forward to the backward. With
 *     dropout_p > 0, sdpa_fwd_ex writes into it the keep bits of every score
 *     tile it computes, and sdpa_bwd_ex, given the same buffer, reads them
 *     instead of drawing them again: the same mask (both sides draw it from
 *     the absolute index, "REDO of dropout support for mem eff #102038",
 *     pytorch PR 103704), so the same results, with the backward's Philox
 *     work replaced by 1/8 byte per score read from device memory. The
 *     backward trusts the buffer: it must be the one the forward filled for
 *     the same B, H, Sq, Sk, dropout_p, seed and offset (or rng_state values)
 *     and batch / head position, unchanged since. Layout: uint32 word
 *     ((b*H + h)*ceil128(Sk)/32 + w)*ceil128(Sq) + i holds the keep bits of
 *     keys 32w .. 32w+31 of query row i (bit e: key 32w+e kept); words of
 *     tiles the causal mask skips are not written. Ignored when dropout_p
 *     is 0. Head dims up to 128 only, without attn_bias and without a packed
 *     batch (else SDPA_ERR_UNSUPPORTED); a short buffer is
 *     SDPA_ERR_INVALID_ARG, a misaligned one SDPA_ERR_ALIGNMENT.
 *   kernel_events: NULL, or a pointer to two cudaEvent_t handles that the
 *     call records on `stream` immediately before and after its main kernel:
 *     the forward kernel, or the backward's main kernel (between its
 *     preprocess and its dQ kernel). A caller times that kernel alone with
 *     cudaEventElapsedTime, without the host work of the call or the
 *     backward's small kernels. Both handles must be non-NULL. Recording is
 *     stream-ordered (under stream capture the records become event-record
 *     nodes of the graph). A call that launches no main kernel (an empty
 *     problem) records neither event.
 */
typedef struct {
  const uint64_t* rng_state;
  int64_t batch_offset;
  int64_t head_offset;
  int64_t total_heads;
  int deterministic;
  const sdpa_tensor* attn_bias;
  sdpa_tensor* dbias;
  void* const* kernel_events;
  uint32_t* dropout_bits;
  size_t dropout_bits_bytes;
} sdpa_options;

/* Bytes of the dropout_bits buffer of a [B, H, Sq, Sk] problem:
 * B*H*ceil128(Sq)*ceil128(Sk)/8 (0 for an empty problem or negative sizes,
 * SIZE_MAX when it does not fit in 62 bits). */
size_t sdpa_dropout_bits_size(int64_t B, int64_t H, int64_t Sq, int64_t Sk);

/* sdpa_fwd with options (NULL options = sdpa_fwd). */
sdpa_status sdpa_fwd_ex(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                        double dropout_p, int is_causal, float scale, uint64_t seed,
                        uint64_t offset, sdpa_tensor* out, float* lse,
                        const sdpa_options* options, sdpa_stream_t stream);

/*
 * sdpa_bwd_workspace_size_ex — workspace bytes of sdpa_bwd_ex with these
 * options: sdpa_bwd_workspace_size(), or in deterministic mode one fp32 dQ
 * slice per 128-key tile, B*H*ceil128(Sq)*(Dk*ceil(Sk/128) + 2)*4 bytes
 * (SIZE_MAX when that does not fit in 62 bits).
 */
size_t sdpa_bwd_workspace_size_ex(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t D,
                                  const sdpa_options* options);

/* sdpa_bwd with options (NULL options = sdpa_bwd); the workspace must have
 * sdpa_bwd_workspace_size_ex() bytes for the same options. */
sdpa_status sdpa_bwd_ex(const sdpa_tensor* dout, const sdpa_tensor* q, const sdpa_tensor* k,
                        const sdpa_tensor* v, const sdpa_tensor* out, const float* lse,
                        double dropout_p, int is_causal, uint64_t seed, uint64_t offset,
                        float scale, sdpa_tensor* dq, sdpa_tensor* dk, sdpa_tensor* dv,
                        void* workspace, size_t workspace_bytes, const sdpa_options* options,
                        sdpa_stream_t stream);

/* sdpa_dropout_mask_debug with options (rng_state and the batch/head
 * position; `deterministic` is ignored). */
sdpa_status sdpa_dropout_mask_debug_ex(int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                                       double dropout_p, uint64_t seed, uint64_t offset,
                                       const sdpa_options* options, uint8_t* mask,
                                       sdpa_stream_t stream);

/*
 * Packed variable-length batches. The fused kernels' forward also reports
 * the maximum query and key lengths (max_q / max_k: "Note to self: Next few
 * PRs" of NVIDIA/Fuser issue 2278, "SdpaOpFwd / SdpaOpBwd nodes"), the
 * sizes of a batch of sequences of different lengths stored back to back.
 * Sequence b of `batch` has query rows [cu_seqlens_q[b], cu_seqlens_q[b+1])
 * of q, out, dout and dq, and key rows [cu_seqlens_k[b], cu_seqlens_k[b+1])
 * of k, v, dk and dv. The tensors are logical [1, H, total, D] (e.g. a
 * packed [total, H, D] buffer viewed with strides (_, D, H*D, 1)), lse is
 * float32 [H, total_q] contiguous. Each sequence is computed as the top-left
 * [len_q, len_k] block of a [max_seqlen_q, max_seqlen_k] problem: causal
 * masking is top-left within the sequence, and the dropout counter uses the
 * padded problem's index, ((b*H + h)*max_seqlen_q + i)*max_seqlen_k + j.
 *   cu_seqlens_q, cu_seqlens_k: device int32 arrays of batch + 1 offsets,
 *     starting at 0, nondecreasing, ending at the tensors' totals. They are
 *     read on the device only, so the host cannot check them; lengths above
 *     the maxima are not allowed. A sequence with queries and no keys gets
 *     out = 0 and lse = -inf.
 *   max_seqlen_q, max_seqlen_k: bounds (>= 1) of the sequences' lengths;
 *     they size the launch grids and the backward workspace.
 * sdpa_options apply as in the *_ex calls, except attn_bias / dbias
 * (SDPA_ERR_UNSUPPORTED with a packed batch).
 */
typedef struct {
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  int64_t batch;
  int64_t max_seqlen_q;
  int64_t max_seqlen_k;
} sdpa_varlen;

sdpa_status sdpa_fwd_varlen(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                            const sdpa_varlen* seqs, double dropout_p, int is_causal, float scale,
                            uint64_t seed, uint64_t offset, sdpa_tensor* out, float* lse,
                            const sdpa_options* options, sdpa_stream_t stream);

/* Workspace bytes of sdpa_bwd_varlen: as sdpa_bwd_workspace_size_ex with B =
 * batch, Sq = max_seqlen_q, Sk = max_seqlen_k. */
size_t sdpa_bwd_varlen_workspace_size(const sdpa_varlen* seqs, int64_t H, int64_t D,
                                      const sdpa_options* options);

sdpa_status sdpa_bwd_varlen(const sdpa_tensor* dout, const sdpa_tensor* q, const sdpa_tensor* k,
                            const sdpa_tensor* v, const sdpa_tensor* out, const float* lse,
                            const sdpa_varlen* seqs, double dropout_p, int is_causal,
                            uint64_t seed, uint64_t offset, float scale, sdpa_tensor* dq,
                            sdpa_tensor* dk, sdpa_tensor* dv, void* workspace,
                            size_t workspace_bytes, const sdpa_options* options,
                            sdpa_stream_t stream);

/*
 * sdpa_check_device — synchronises `stream`, then reports whether any kernel
 * of this library on the current device gave up on a bounded wait since the
 * last check (SDPA_ERR_DEVICE_TIMEOUT; the word is cleared) or the stream
 * reported a CUDA error (SDPA_ERR_CUDA). The pages have no counterpart: this
 * is the library's failure-detection hook.
 */
sdpa_status sdpa_check_device(sdpa_stream_t stream);

/*
 * sdpa_selftest_wait_timeout — launches one tiny kernel that waits, with the
 * given bound in nanoseconds, on an mbarrier that nothing ever arrives on,
 * then synchronises and returns SDPA_ERR_DEVICE_TIMEOUT if the wait gave up
 * as designed (SDPA_OK would mean the barrier completed, which cannot
 * happen). It exercises the bounded-wait path without faulting or hanging
 * the GPU. No counterpart on the pages.
 */
sdpa_status sdpa_selftest_wait_timeout(uint64_t limit_ns, sdpa_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* sdpa_status_string(sdpa_status status);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_GB300_H */
