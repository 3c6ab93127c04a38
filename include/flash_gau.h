/*
 * flash_gau.h -- C ABI of libflashgau, the sm_103a (GB300) forward pass of
 * the FLASH gated attention unit with mixed chunk attention.
 *
 * The operation ("Transformer Quality in Linear Time", Method, eq. 5, eq. 7,
 * eq. 8 and the display after eq. 8; "FLASH: Possibly the Most Interesting
 * Efficient Transformer Design in Recent Times", sections "Gated Attention",
 * "Weak Attention" and "Mixed Chunking"):
 *
 *   [U | V | Z] = swish(X [W_u | W_v | W_z])               swish(x) = x*sigmoid(x)
 *   Q_quad, K_quad, Q_lin, K_lin = Z * gamma_h + beta_h     (per-dimension heads)
 *   for every chunk g of C consecutive tokens (G = T / C chunks):
 *     Vq_g   = local_scale * relu^2(Q_quad,g K_quad,g^T / C + b) V_g
 *                                                          b[i][j] = relpos[j-i+C-1]
 *              (entries with j > i are zero when causal; diagonal kept)
 *     P_g    = sum_{h<g} K_lin,h^T V_h   (causal, eq. 8; zero for g = 0)
 *            = sum_{h}   K_lin,h^T V_h   (non-causal, eq. 7)
 *     Vl_g   = lin_scale * Q_lin,g P_g
 *     O_g    = [U_g * (Vq_g + Vl_g)] W_o
 *
 * Readings where the pages differ: scores are divided by C before the bias
 * (flash_block pseudocode); the chunk states are summed plainly (eq. 7/8),
 * lin_scale = 1 reproduces that, 1/C the appendix listing, 0 the LocalOnly
 * ablation; local_scale = 1 is the layer as written, 0 the GlobalOnly
 * ablation (section 4.4: only the global, linear part); the Toeplitz bias of appendix D Code 4 (2C-1 weights) is used for
 * every C.  No projection biases, norm, RoPE or residual are applied.
 *
 * Conventions for every entry point:
 *   - Pointers named "device" are CUDA device pointers on the current device;
 *     the caller owns every buffer.  The library allocates no memory.
 *   - All matrices are dense and row-major (last index fastest), without
 *     padding between rows.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Calls are asynchronous: they return once the kernels are
 *     queued, and the caller synchronises.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns a negative status and enqueues nothing.  No C++
 *     exception crosses this interface.
 *   - Entry points are thread-safe with respect to one another, except that
 *     concurrent forwards must not share a workspace.
 */
#ifndef FLASH_GAU_H
#define FLASH_GAU_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define FLASH_GAU_OK 0
#define FLASH_GAU_EINVAL (-1)     /* null pointer, bad size, T % C != 0, ... */
#define FLASH_GAU_ENOTSUP (-2)    /* valid shape outside the supported set   */
#define FLASH_GAU_EWORKSPACE (-3) /* workspace too small or misaligned       */
#define FLASH_GAU_ECUDA (-4)      /* CUDA runtime/launch error (see strerror) */
#define FLASH_GAU_EDEVICE (-5)    /* current device is not sm_103            */
#define FLASH_GAU_ETIMEOUT (-6)   /* a kernel gave up a bounded wait         */

/* ---- io data types ----------------------------------------------------- */
/* FP32: X, weights, out and all intermediates in fp32, fp32 arithmetic.
 * BF16: X, W_uvz, W_o and out in bf16; tensor-core products with fp32
 *       accumulation; U, V, heads, chunk states, prefix states and the gated
 *       product are stored in bf16 (prefix sums accumulate in fp32).
 *       gamma, beta and relpos are fp32 for both types.                     */
#define FLASH_GAU_FP32 0
#define FLASH_GAU_BF16 1

typedef struct flash_gau_weights {
  const void *W_uvz;    /* device [d, 2e+s], io type: columns [0,e) W_u,
                           [e,2e) W_v, [2e,2e+s) W_z                        */
  const void *W_o;      /* device [e, d], io type                           */
  const float *gamma;   /* device [4, s] fp32, rows Q_quad K_quad Q_lin K_lin */
  const float *beta;    /* device [4, s] fp32, same row order               */
  const float *relpos;  /* device [2C-1] fp32, b[i][j] = relpos[j-i+C-1]    */
  int d;                /* model width                                      */
  int e;                /* expansion width (U, V)                           */
  int s;                /* shared head width (Z)                            */
  float lin_scale;      /* factor on the global (linear) term               */
  float local_scale;    /* factor on the local (quadratic) term: 1 as
                           written; 0 skips the chunk scores entirely       */
} flash_gau_weights;

/* Byte offsets of the intermediates inside a workspace (all from its start).
 * io = the io type's size.  The offsets are 256-byte aligned.              */
typedef struct flash_gau_workspace_layout {
  size_t total_bytes;   /* bytes the workspace must hold                    */
  size_t status;        /* int32 device status word (FLASH_GAU_ETIMEOUT...);
                           the rest of its 256-byte slot is used by the
                           kernels for scheduling                            */
  size_t U;             /* [B*T, e] io: swish(X W_u)                        */
  size_t V;             /* [B*T, e] io: swish(X W_v)                 (*)    */
  size_t heads;         /* [4, B*T, s] io: Q_quad, K_quad, Q_lin, K_lin      */
  size_t state;         /* [B, G, s, e] io: K_lin,g^T V_g per chunk   (*)    */
  size_t prefix;        /* [B, G, s, e] io: lin_scale * (exclusive / total)
                           chunk-state sum of each chunk; a non-causal
                           forward without segments writes only the first
                           [B, s, e] (one total per batch row)        (*)   */
  size_t gated;         /* [B*T, e] io: U * (Vq + Vl)                       */
  size_t bias;          /* [2C-1] fp32: relpos as the bf16 attention kernel
                           reads it; causal: the entries of offset j-i >= 1
                           are -inf, so relu^2 applies the causal mask      */
  size_t xn;            /* [B*T, d] io: the normalised input of
                           flash_gau_block_forward (unused otherwise)       */
  size_t rope;          /* [s/2, T] fp16 (cos, sin) pairs: the RoPE table of
                           flash_gau_block_forward, bf16 (unused otherwise) */
} flash_gau_workspace_layout;
/* Intermediates are row-major, except those marked (*) for FLASH_GAU_BF16:
 * these, seen as [rows, e] matrices (rows = B*T, B*G*s or B*s), are stored
 * in 64 x 64 blocks, row-block-major: block (i, j) holds rows 64i..64i+63
 * and columns 64j..64j+63 as 8 KB of row-major data, at block index
 * i * (e / 64) + j.  Element (r, c) is at offset
 * ((r / 64) * (e / 64) + c / 64) * 4096 + (r % 64) * 64 + c % 64.          */

/* Supported shapes.  All types: B, T, C, d, e, s > 0 and T % C == 0.
 *   FP32: any such shape with s <= 128 and C <= 4096.
 *   BF16: d % 128 == 0, e % 256 == 0, s == 128, C % 128 == 0, C <= 4096.
 * Other shapes return FLASH_GAU_ENOTSUP.                                   */

/* Fills *out for the given problem.  Returns FLASH_GAU_OK, FLASH_GAU_EINVAL
 * (bad sizes or null out) or FLASH_GAU_ENOTSUP.                            */
int flash_gau_workspace_layout_query(int B, int T, int C, int d, int e, int s,
                                     int causal, int dtype,
                                     flash_gau_workspace_layout *out);

/* Workspace size in bytes for the given problem, or 0 if the arguments are
 * invalid or unsupported.                                                  */
size_t flash_gau_workspace_bytes(int B, int T, int C, const flash_gau_weights *w,
                                 int causal, int dtype);

/* The forward pass, O = FLASH-GAU(X).
 *   X         device [B, T, d], io type
 *   w         host pointer to the weight descriptor (read during the call)
 *   B, T, C   batch, sequence length, chunk length (T % C == 0; C == T gives
 *             FLASH-Quad, the quadratic GAU)
 *   causal    nonzero: causal local mask and exclusive chunk prefix (eq. 8);
 *             zero: full local attention and total chunk sum (eq. 7)
 *   dtype     FLASH_GAU_FP32 or FLASH_GAU_BF16
 *   out       device [B, T, d], io type; must not overlap X or the workspace
 *   workspace device, >= flash_gau_workspace_bytes(...) bytes, 256-byte
 *             aligned; its contents on return are the intermediates listed
 *             in flash_gau_workspace_layout
 *   stream    cudaStream_t
 * Returns FLASH_GAU_OK once all kernels are queued, or a negative status.  A
 * kernel that gives up a bounded wait records FLASH_GAU_ETIMEOUT in the
 * workspace status word; read it with flash_gau_workspace_status().        */
int flash_gau_forward(const void *X, const flash_gau_weights *w, int B, int T,
                      int C, int causal, int dtype, void *out, void *workspace,
                      size_t workspace_bytes, void *stream);

/* Same as flash_gau_forward, and additionally records stage_events[0] on the
 * stream before the first kernel and stage_events[k+1] after stage k
 * (k = 0 .. n_events-2).  stage_events are cudaEvent_t handles owned by the
 * caller; n_events may be 0.  The stage count and names come from
 * flash_gau_num_stages / flash_gau_stage_name.                              */
int flash_gau_forward_timed(const void *X, const flash_gau_weights *w, int B,
                            int T, int C, int causal, int dtype, void *out,
                            void *workspace, size_t workspace_bytes,
                            void *stream, void *const *stage_events,
                            int n_events);

/* Number of kernel stages one forward launches for this dtype / causality,
 * and a static name for stage k (NULL when out of range).                  */
int flash_gau_num_stages(int dtype, int causal);
const char *flash_gau_stage_name(int dtype, int causal, int k);

/* Synchronises `stream`, returns the status word the kernels left in the
 * workspace (FLASH_GAU_OK or FLASH_GAU_ETIMEOUT) and resets it to zero.
 * Returns FLASH_GAU_ECUDA if the stream reported an error.                 */
int flash_gau_workspace_status(void *workspace, void *stream);

/* Static description of a status code.  For FLASH_GAU_ECUDA it includes the
 * last CUDA error seen by this thread.                                     */
const char *flash_gau_strerror(int status);

/* Library version as major*10000 + minor*100 + patch.                      */
int flash_gau_version(void);

/* ---- the flash_block wrapper -------------------------------------------- */
/* The block around the layer in the pages' flash_block pseudocode
 * ("Transformer Quality in Linear Time", flash_block; gau_block has the same
 * frame):  Y = X + layer(norm(X)),  where the layer's four heads are rotated
 * by RoPE at the tokens' global positions before use.  The pages print
 * neither the norm nor the rope function; this library's readings:
 *   LayerNorm  (x - mean) / sqrt(var + eps) * g + b   (biased variance)
 *   ScaleNorm  g * x / max(||x||_2, eps)              (g a single scalar)
 *   RoPE       the pair (h[2i], h[2i+1]) of a head of the token at position
 *              p = t + pos_offset (t its index in its sequence) is rotated
 *              by the angle p * rope_base^(-2i/s).                          */
#define FLASH_GAU_NORM_NONE 0
#define FLASH_GAU_NORM_LAYER 1
#define FLASH_GAU_NORM_SCALE 2

typedef struct flash_gau_block {
  int norm;             /* FLASH_GAU_NORM_NONE / _LAYER / _SCALE             */
  const float *norm_g;  /* device fp32: LayerNorm scale [d], ScaleNorm g [1] */
  const float *norm_b;  /* device fp32: LayerNorm shift [d], or NULL (zero)  */
  float norm_eps;       /* > 0                                               */
  int rope;             /* nonzero: rotate the four heads (s must be even)   */
  float rope_base;      /* > 1 (10000 in the rotary embedding's definition)  */
  int pos_offset;       /* >= 0: position of each sequence's first token     */
  int residual;         /* nonzero: add X (the shortcut) to the output       */
} flash_gau_block;

/* Y = [X +] layer(norm(X)) with RoPE on the heads, per the options in *blk
 * (host pointer, read during the call).  The other arguments, the
 * workspace and the status word are as for flash_gau_forward; the workspace
 * region xn holds the normalised input.  blk->norm == NONE, rope == 0 and
 * residual == 0 compute exactly flash_gau_forward.  Returns FLASH_GAU_EINVAL
 * for bad options (unknown norm, missing norm_g, eps <= 0, rope with an odd
 * s or base <= 1, negative pos_offset).                                      */
int flash_gau_block_forward(const void *X, const flash_gau_weights *w,
                            const flash_gau_block *blk, int B, int T, int C,
                            int causal, int dtype, void *out, void *workspace,
                            size_t workspace_bytes, void *stream);

/* ---- diagnostics -------------------------------------------------------- */
/* Checks that a wait the library's kernels make gives up instead of hanging:
 * one kernel waits on something that nothing signals, then records
 * FLASH_GAU_ETIMEOUT.  which = 0 waits on a shared-memory mbarrier (the form
 * of the TMA and tensor-core pipelines), 1 on a flag in global memory (the
 * form of the chunk-state kernel's grid barrier).  words: device int[2],
 * zeroed by the caller; once the stream has run the kernel (about two
 * seconds, the library's wait limit) words[0] holds FLASH_GAU_ETIMEOUT and
 * the context stays usable.  Returns FLASH_GAU_OK once queued, or
 * FLASH_GAU_EINVAL.                                                        */
int flash_gau_selftest_bounded_wait(int which, int *words, void *stream);

/* ---- host buffers ----------------------------------------------------- */
/* The forward pass on host memory: X_host [B, T, d] is copied to the
 * device, the layer runs, and O is copied back to out_host [B, T, d] (both
 * io type, host pointers; page-locked memory lets the copies run
 * asynchronously and overlap, pageable memory works but copies
 * synchronously).  Batch rows are independent, so the batch is cut into up
 * to four parts: the input copy of one part, the layer on another and the
 * output copy of a third run at the same time.  The copies run on two
 * streams that the library creates once per device (no device memory) and
 * shares between calls; the layer runs on `stream`, which is made to wait
 * for the last output copy before the call returns, and whose earlier work
 * comes first.  Synchronise `stream` before reading out_host.  Calls on
 * one device are serialised while they enqueue.
 *   workspace  device, >= flash_gau_forward_host_workspace_bytes(...)
 *              bytes, 256-byte aligned: device copies of X and O, then the
 *              layer's workspace for one part of the batch
 * Other arguments and return values as for flash_gau_forward.             */
size_t flash_gau_forward_host_workspace_bytes(int B, int T, int C,
                                              const flash_gau_weights *w,
                                              int causal, int dtype);
int flash_gau_forward_host(const void *X_host, const flash_gau_weights *w,
                           int B, int T, int C, int causal, int dtype,
                           void *out_host, void *workspace,
                           size_t workspace_bytes, void *stream);

/* ---- segment masks (packed text) -------------------------------------- */
/* The global term with a chunk mask ("Transformer Quality in Linear Time",
 * Paper vs code, the segment-mask item; Pitfalls, the same item): segment
 * ids mask the chunk summaries in the linear part only (the local part is
 * unchanged), and each row of the mask may be normalised to sum to one, so
 * the global term becomes the mean of the visible chunk states:
 *   Prefix_g = lin_scale * sum_h M[g, h] State_h
 *   M[g, h]  = 1 when h is visible from g (h < g causal, any h otherwise)
 *              and g, h lie in one segment; rows divided by their count
 *              when `average` (an empty row stays zero).
 * Reading: a segment is a maximal run of consecutive chunks with one id (a
 * change of id between neighbouring chunks starts a new segment; packed
 * text gives each document one run, whole chunks each).                   */
typedef struct flash_gau_segments {
  const int *ids;  /* device [B, G] int32 chunk segment ids, or NULL (the
                      whole sequence is one segment)                       */
  int average;     /* nonzero: row-normalised mask (mean of the states)    */
} flash_gau_segments;

/* flash_gau_forward with the chunk mask of `seg` (a host pointer, read
 * during the call; NULL = no mask, the plain sums of eq. 7/8).  Arguments
 * and workspace as for flash_gau_forward.                                  */
int flash_gau_forward_segmented(const void *X, const flash_gau_weights *w,
                                const flash_gau_segments *seg, int B, int T,
                                int C, int causal, int dtype, void *out,
                                void *workspace, size_t workspace_bytes,
                                void *stream);

/* ---- backward pass ------------------------------------------------------ */
/* Gradients of L = sum(dO * O), O = flash_gau_forward(X, ...), with respect
 * to X and every parameter, by the chain rule through the forward's steps
 * (eq. 5, eq. 7, eq. 8 and the display after it): the backward the pages'
 * training workloads need.  The call recomputes the forward's
 * intermediates itself (it needs no earlier forward).  For bf16 io with
 * B*T, d, e, C and s multiples of 128 every contraction runs on the
 * tcgen05 tensor cores with bf16 operands and fp32 accumulation (with C or
 * s not multiples of 128, the chunk-level ones run on the CUDA cores);
 * fp32 io, and other bf16 shapes, run the contractions in fp32 on the
 * CUDA cores.  Sums and scans are fp32 in both cases; on the tensor-core
 * path the elementwise steps run in fp32 on bf16 operands, most of them in
 * the epilogues of the contractions.  Gradients are written, not added.    */
typedef struct flash_gau_grads {
  void *dX;          /* device [B, T, d], io type                           */
  float *dW_uvz;     /* device [d, 2e+s] fp32, columns as in W_uvz          */
  float *dW_o;       /* device [e, d] fp32                                  */
  float *dgamma;     /* device [4, s] fp32                                  */
  float *dbeta;      /* device [4, s] fp32                                  */
  float *drelpos;    /* device [2C-1] fp32                                  */
} flash_gau_grads;

/* fp32 work-buffer bytes flash_gau_backward needs, or 0 when the arguments
 * are invalid or unsupported (B*T > 65535*64, B*T/C > 65535, C > 4096).   */
size_t flash_gau_backward_workspace_bytes(int B, int T, int C,
                                          const flash_gau_weights *w,
                                          int causal, int dtype);

/* X and dO: device [B, T, d], io type; w as for the forward (lin_scale
 * included); g: host pointer to the gradient outputs; workspace: device,
 * 256-byte aligned, >= flash_gau_backward_workspace_bytes.  Enqueued on
 * `stream`, no synchronisation.  Returns FLASH_GAU_OK, FLASH_GAU_EINVAL,
 * FLASH_GAU_ENOTSUP, FLASH_GAU_EWORKSPACE or FLASH_GAU_ECUDA.            */
int flash_gau_backward(const void *X, const void *dO, const flash_gau_weights *w,
                       int B, int T, int C, int causal, int dtype,
                       const flash_gau_grads *g, void *workspace,
                       size_t workspace_bytes, void *stream);

/* ---- autoregressive decode ---------------------------------------------- */
/* One new token for each of B sequences, in constant work per token
 * (Transformer Quality in Linear Time §3.2.1: the global term is carried as
 * one running matrix and the local attention reaches back within the
 * current chunk only).  The state, one
 * buffer per batch of sequences, keeps per sequence the number of tokens
 * consumed, the linear cache (the sum of K_lin^T V over its completed
 * chunks, fp32 [s, e]) and the current chunk's K_quad, K_lin and V rows
 * (fp32).  A zeroed state starts B new sequences at position 0; each call
 * consumes token x[b] of every sequence and writes its output, the row the
 * causal forward would give it.  Each call enqueues five kernels on
 * `stream` and does not synchronise.                                       */

/* State bytes for B sequences, or 0 when the arguments are invalid or
 * unsupported (B <= 65535, C <= 4096, s <= 256, d and e <= 16384, d, e and
 * s multiples of 8).                                                       */
size_t flash_gau_decode_state_bytes(int B, int C, const flash_gau_weights *w,
                                    int dtype);

/* x, out: device [B, d], io type; state: device, 256-byte aligned,
 * >= flash_gau_decode_state_bytes; w as for the forward (causal).  Returns
 * FLASH_GAU_OK, FLASH_GAU_EINVAL, FLASH_GAU_ENOTSUP, FLASH_GAU_EWORKSPACE
 * or FLASH_GAU_ECUDA.                                                      */
int flash_gau_decode_step(const void *x, const flash_gau_weights *w, int B, int C,
                          int dtype, void *state, size_t state_bytes, void *out,
                          void *stream);

/* ---- RoPE construction of the relative position bias ------------------- */
/* Appendix D, Code 4 of "Transformer Quality in Linear Time" builds the bias
 * of windows of 512 positions and more from two learned vectors a, b of
 * width m (128 there): both are tiled over the window, each row rotated by
 * RoPE at its position, and bias[i][j] = rope(a)_i . rope(b)_j.  Rotations
 * compose, so the matrix depends on j - i only; this call writes it in the
 * layer's table form, relpos[j - i + C - 1] (2C - 1 fp32 values), ready to
 * pass as flash_gau_weights.relpos.
 *   a, b       device fp32 [m], m even, 2 <= m <= 128
 *   C          window (chunk) length, 1 <= C <= 4096
 *   rope_base  > 1; the pair (2k, 2k+1) turns by p * rope_base^(-2k/m)
 *   relpos     device fp32 [2C - 1], written
 * Enqueued on `stream`, no synchronisation.  Returns FLASH_GAU_OK,
 * FLASH_GAU_EINVAL (null pointer or sizes out of range) or FLASH_GAU_ECUDA. */
int flash_gau_rope_toeplitz_bias(const float *a, const float *b, int m, int C,
                                 float rope_base, float *relpos, void *stream);

/* ---- allocation-free variant ------------------------------------------- */
/* No counterpart on the pages: this entry point exists for deployment, not
 * for the method.
 *
 * Some callers cannot allocate device memory at the point where they run
 * the layer: a plugin whose host framework owns every byte of the device
 * through its own pool and forbids raw allocations, a callback that runs
 * while such a pool is locked, or a latency-critical path that must not
 * take the implicit device synchronisation of cudaMalloc/cudaFree.  For
 * them, flash_gau_forward_noalloc computes exactly what flash_gau_forward
 * computes, but keeps its intermediates in a scratch array that is part of
 * the library image instead of a caller-supplied workspace.
 *
 *   - The scratch is a file-scope static __device__ array of
 *     FLASH_GAU_NOALLOC_SCRATCH_BYTES (32 MiB).  Every GPU on which the
 *     library's device code is loaded holds these 32 MiB until the process
 *     exits.
 *   - Problems whose workspace (flash_gau_workspace_bytes) is larger than
 *     the scratch are rejected with FLASH_GAU_EWORKSPACE before anything is
 *     launched; other argument errors return the same codes as
 *     flash_gau_forward.  Every check runs before the array is touched, so
 *     a rejected call leaves it (and its status word) as it was.
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and caches it; make
 *     that first call before any stream capture on that device.  The
 *     cached address is not looked up again, so resetting a device
 *     (cudaDeviceReset) while the library stays loaded is not supported.
 *   - The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 *     library routine.  It enqueues a 4-byte cudaMemsetAsync that clears
 *     the status word, then the same kernels as flash_gau_forward, on
 *     `stream`, and returns without synchronising.
 *   - All calls on a device share the one array, which keeps the previous
 *     call's intermediates.  Calls whose kernels overlap on the GPU (other
 *     streams, other host threads) race on it: the caller must order them,
 *     e.g. by issuing them on one stream.
 *   - A bounded-wait timeout of these kernels is recorded in the shared
 *     status word only and is not reported to the caller.
 * Arguments as for flash_gau_forward, without the workspace.               */
#define FLASH_GAU_NOALLOC_SCRATCH_BYTES ((size_t)32 * 1024 * 1024)
int flash_gau_forward_noalloc(const void *X, const flash_gau_weights *w, int B, int T,
                              int C, int causal, int dtype, void *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FLASH_GAU_H */
