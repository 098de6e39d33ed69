/*
 * tm.h -- C ABI of libtm, the B300 (sm_103a) triangle multiplicative update.
 *
 * The operation. The pages name the layer -- TriangleMultiplicationOutgoing,
 * built once on the CPU and applied as layer(x, mask), with an Outgoing
 * direction selector, in the code-sample section ("Exemplo de código: triangle
 * multiplication CP-aware") of "NVIDIA BioNeMo escala modelagem biomolecular com
 * context parallelism e quebra barreira de memória da GPU" -- and work it over
 * the N x N pair representation of that page's "2D tiling da pair
 * representation" section, but they do not write its arithmetic out. libtm
 * computes the standard AlphaFold3/Boltz Pairformer definition over z [N][N][c_z]:
 *
 *   zh_ij  = LayerNorm_in(z_ij)                              over c_z, eps 1e-5
 *   a_ik   = sigmoid(W_ga zh_ik) * (W_a zh_ik) * m_i m_k     c_h channels
 *   b_ik   = sigmoid(W_gb zh_ik) * (W_b zh_ik) * m_i m_k
 *   x_ij   = sum_k a_ik b_jk      (TM_OUTGOING)
 *   x_ij   = sum_k a_ki b_kj      (TM_INCOMING)
 *   out_ij = sigmoid(W_g zh_ij) * W_o LayerNorm_out(x_ij)    LayerNorm over c_h
 *
 * m is a token mask [N] of 0/1 values; Linear layers have no bias; LayerNorm
 * uses the biased variance.
 *
 * Precisions. TM_BF16: z and out are bf16, a and b are stored as bf16
 * channel-major [c_h][N][ld]; x, on its way from the contraction to the output
 * LayerNorm, is fp16 scaled by one power of two 2^e by default (tm_x_storage
 * below) and float32 with TM_X_FP32; every contraction accumulates in float32
 * on the tensor cores (tcgen05); c_z = c_h = 128 only. TM_F32: z, out and every
 * intermediate are float32, computed with FP32 FMA on the CUDA cores; any
 * 1 <= c_z, c_h <= 256.
 *
 * Conventions for every call below.
 *  - Pointers named "device" are device memory of the ctx's GPU; "host" ones
 *    are host memory. Tensors are dense, row-major, 16-byte aligned.
 *  - The caller owns z, mask and out; libtm owns its workspace (a, b and a
 *    block of x), grows it with cudaMallocAsync on the call's stream, and frees
 *    it in tm_destroy.
 *  - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t,
 *    NULL for the legacy default stream). Argument errors return
 *    synchronously, before any launch. A device-side wait that exceeds its
 *    time limit stores TM_ERR_TIMEOUT in the ctx's status word; the next
 *    tm_forward* or tm_sync_status returns it.
 *  - A ctx may be used from one host thread and one stream at a time.
 */
#ifndef TM_H
#define TM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tm_ctx tm_ctx; /* opaque, owned by libtm */

typedef enum {
  TM_OK = 0,
  TM_ERR_INVALID = 1,     /* bad pointer, size, alignment, aliasing or enum value      */
  TM_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. bf16 with c != 128)       */
  TM_ERR_OOM = 3,         /* workspace would exceed the limit, or allocation failed    */
  TM_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (see tm_last_error)     */
  TM_ERR_TIMEOUT = 5      /* a device-side wait ran out of time (status word)          */
} tm_status;

typedef enum { TM_OUTGOING = 0, TM_INCOMING = 1 } tm_direction;
typedef enum { TM_F32 = 0, TM_BF16 = 1 } tm_dtype;

/* Layer parameters: host float32 arrays, Linear layout [out][in] (y = W x). */
typedef struct {
  const float *ln_in_gamma, *ln_in_beta;   /* [c_z]        */
  const float *w_a, *w_ga, *w_b, *w_gb;    /* [c_h][c_z]   */
  const float *w_g;                        /* [c_z][c_z]   */
  const float *ln_out_gamma, *ln_out_beta; /* [c_h]        */
  const float *w_o;                        /* [c_z][c_h]   */
} tm_weights;

/* Storage of the contraction's output x (c_h values per pair of the current
 * output block) on its way to the output LayerNorm, bf16 path only:
 *   TM_X_FP16  fp16, every value scaled by one power of two 2^e with
 *              e = 14 - ceil(log2(N max_c(A_c B_c))) (clamped to [-60, 60]),
 *              A_c = sqrt(c_z) ||W_a[c] diag(gamma_in)|| + |(W_a beta_in)_c|
 *              bounding |a_c| for any input (B_c likewise for b); since
 *              |x_ij^c| <= N max|a_c| max|b_c|, no value can overflow, and
 *              LayerNorm (scale-free but for its epsilon, which is scaled
 *              alike) reads the scaled values as they are;
 *   TM_X_FP32  float32.
 * The float32 path always keeps x in float32. */
typedef enum { TM_X_FP16 = 0, TM_X_FP32 = 1 } tm_x_storage;

typedef struct {
  int block;              /* edge of the square output blocks of the streamed
                             schedule; 0 = automatic (whole grid while its x
                             fits the workspace limit, else about 2500)            */
  int timeout_ms;         /* limit of every device-side wait; 0 = 2000 ms           */
  size_t workspace_limit; /* bytes; 0 = env TM_WORKSPACE_LIMIT, else no limit      */
  int x_storage;          /* tm_x_storage; 0 = TM_X_FP16                            */
  int residual;           /* 1: out = z + update, the residual connection of a
                             Pairformer block (bf16: one rounding of the sum, as a
                             bf16 add does); out may then be z itself (in place,
                             no extra pass) or a separate buffer (z is copied into
                             it first). 0: out = update, out must not overlap z.  */
  int reserved[6];        /* must be zero                                          */
} tm_options;

/* Create a context on the current CUDA device. Copies and converts the
 * weights (host float32, freed by the caller at will) into the device layouts
 * of both precisions. Returns TM_ERR_INVALID for a NULL argument or c_z, c_h
 * outside [1, 256]. *out_ctx is set only on TM_OK. Synchronous. */
tm_status tm_create(int c_z, int c_hidden, const tm_weights* w, tm_ctx** out_ctx);

/* One triangle multiplicative update: out = update(z, mask) in direction dir.
 *   z     device, [N][N][c_z] of dtype;
 *   mask  device float32 [N] of 0/1 token-mask values, or NULL for all ones;
 *   N     >= 1 tokens;
 *   out   device, [N][N][c_z] of dtype; must not overlap z.
 * The pages' "layer(x, mask)" call of the code-sample section named above. */
tm_status tm_forward(tm_ctx* ctx, const void* z, const float* mask, int N, tm_dtype dtype,
                     tm_direction dir, void* out, void* stream);

/* tm_forward with options (NULL = defaults). */
tm_status tm_forward_ex(tm_ctx* ctx, const void* z, const float* mask, int N, tm_dtype dtype,
                        tm_direction dir, void* out, void* stream, const tm_options* opt);

/* The two triangle multiplicative updates of a Pairformer block, in place:
 *   z <- z + update_outgoing(z);  z <- z + update_incoming(z)
 * (the residual connections around the two layers; "outgoing then incoming,
 * as in one Pairformer block" of the four-chain complex workload). z is
 * device [N][N][c_z] of dtype and is overwritten; each update is a
 * tm_forward_ex with residual = 1 and out = z, so the sums are formed where
 * the finish kernel writes (no extra pass over z). opt as for tm_forward_ex
 * (residual is ignored; NULL = defaults). Stream-ordered; capturable into a
 * CUDA graph once a first call has sized the workspace. */
tm_status tm_pair_update(tm_ctx* ctx, void* z, const float* mask, int N, tm_dtype dtype, void* stream,
                         const tm_options* opt);

/* tm_forward on HOST buffers: copies z (and mask) host -> device into
 * ctx-owned device buffers, runs the update, and copies out device -> host;
 * returns after enqueueing (synchronise `stream` before reading out).
 *   z_host     host [N][N][c_z] of dtype (page-locked memory lets the copies
 *              run asynchronously; pageable memory works but blocks);
 *   mask_host  host float32 [N] or NULL;
 *   out_host   host [N][N][c_z] of dtype.
 * The copies run on two streams of the ctx, ordered against `stream` by
 * events, through two device staging slots that calls use in turn: a call's
 * copy in may run while the call before it still computes or copies back, the
 * kernels run on `stream` after the copy in, and for bf16 the output leaves in
 * strips of 512 rows, each as soon as its rows are finished, while the next
 * strip computes; at the end `stream` waits for the copy back. z_host must
 * hold its values when the call is made (a z_host that overlaps the previous
 * call's out_host is copied after that call's copy back). The device staging
 * (twice z and out) is owned by the ctx and freed by tm_destroy. */
tm_status tm_forward_host(tm_ctx* ctx, const void* z_host, const float* mask_host, int N,
                          tm_dtype dtype, tm_direction dir, void* out_host, void* stream);

/* The three steps of tm_forward, for callers that keep intermediates. The
 * plain forms (tm_project, tm_contract, tm_finish) run the float32-x variant
 * (tm_forward_ex with x_storage = TM_X_FP32); the _ex forms also run the
 * default fp16 x, and tm_project_ex -> tm_contract_ex -> tm_finish_ex over the
 * whole grid with TM_X_FP16 gives tm_forward's result bit for bit.
 *
 * tm_project: a, b = gated, masked projections of LayerNorm(z).
 *   a, b  device, channel-major [c_h][N][ld] of dtype (bf16 or float32);
 *   ld    >= N, and a multiple of 8 for TM_BF16 (16-byte rows).
 */
tm_status tm_project(tm_ctx* ctx, const void* z, const float* mask, int N, tm_dtype dtype,
                     void* a, void* b, int ld, void* stream);

/* tm_project that also writes, per pair, the LayerNorm_in statistics that the
 * fp16-x finish step reads:
 *   zstat  device float32 [N][N][2] = (rstd, -rstd * mean) of z_ij over c_z, or
 *          NULL (not written); 8-byte aligned; TM_BF16 only. */
tm_status tm_project_ex(tm_ctx* ctx, const void* z, const float* mask, int N, tm_dtype dtype,
                        void* a, void* b, int ld, float* zstat, void* stream);

/* The exponent e of the fp16 storage of x for a grid of N tokens: every x value
 * is stored times 2^e (the bound in the tm_x_storage comment). 0 for a NULL ctx
 * or one without the bf16 path. */
int tm_x_exponent(const tm_ctx* ctx, int N);

/* tm_contract: the per-channel contraction over one output block.
 *   a, b    device, [c_h][N][ld] of dtype, as written by tm_project;
 *   i0, j0  first row / column of the block; bi, bj its extents (>= 1);
 *   x       device float32 [c_h][bi][ldx], ldx >= bj and a multiple of 4;
 *           x[c][i - i0][j - j0] = sum_k a.. b.. as in the header comment.
 *           Columns [bj, roundup(bj, 4)) of each row may be overwritten (the
 *           stores move whole 16-byte granules); nothing past them is.
 */
tm_status tm_contract(tm_ctx* ctx, const void* a, const void* b, int N, int ld, tm_dtype dtype,
                      tm_direction dir, int i0, int j0, int bi, int bj, float* x, int ldx,
                      void* stream);

/* tm_contract with the storage of x chosen: x_storage TM_X_FP32 as tm_contract;
 * TM_X_FP16 (TM_BF16 only) writes x as fp16 times 2^tm_x_exponent(ctx, N) into
 * x [c_h][bi][ldx] with ldx >= bj and a multiple of 8; only columns < bj of
 * each row are written. */
tm_status tm_contract_ex(tm_ctx* ctx, const void* a, const void* b, int N, int ld, tm_dtype dtype,
                         tm_direction dir, int i0, int j0, int bi, int bj, void* x, int ldx,
                         int x_storage, void* stream);

/* tm_finish: out over one block from its x block and z.
 *   x    device float32 [c_h][bi][ldx] (as tm_contract writes it);
 *   z    device [N][N][c_z] of dtype;
 *   out  device [N][N][c_z] of dtype; only entries of the block are written.
 */
tm_status tm_finish(tm_ctx* ctx, const float* x, int ldx, const void* z, int N, tm_dtype dtype,
                    int i0, int j0, int bi, int bj, void* out, void* stream);

/* tm_finish with the storage of x chosen: x as tm_contract_ex wrote it with the
 * same x_storage; TM_X_FP16 also needs zstat as tm_project_ex wrote it for the
 * same z (TM_ERR_INVALID without it). */
tm_status tm_finish_ex(tm_ctx* ctx, const void* x, int ldx, int x_storage, const float* zstat,
                       const void* z, int N, tm_dtype dtype, int i0, int j0, int bi, int bj,
                       void* out, void* stream);

/* The steps of the update on one block of a pair representation that is split into square blocks
 * across devices (the 2D tiling of the "2D tiling da pair representation" section of the BioNeMo
 * context-parallelism page named above; pair_representation_boltz_b300/ring2d.py schedules them). A block
 * covers B row tokens I and B column tokens K; its token masks differ between rows and columns.
 *
 * tm_project_block: a, b of the block: a_ik = sigmoid(W_ga zh_ik) (W_a zh_ik) m_i m_k over i in I, k in K.
 *   z          device bf16 [B][B][c_z], the block;
 *   mask_rows  device float32 [B] token mask of I, or NULL (ones);
 *   mask_cols  device float32 [B] token mask of K, or NULL (ones);
 *   a, b       device bf16 [c_h][B][ld], ld >= B and a multiple of 8;
 *   zstat      as for tm_project_ex, or NULL.
 * TM_BF16 (c_z = c_h = 128) only. */
tm_status tm_project_block(tm_ctx* ctx, const void* z, const float* mask_rows, const float* mask_cols, int B,
                           void* a, void* b, int ld, float* zstat, void* stream);

/* The contraction of one pair of B x B operand blocks into a float32 x block:
 *   TM_OUTGOING  x[c][i][j] (+)= sum_k a[c][i][k] b[c][j][k]
 *   TM_INCOMING  x[c][i][j] (+)= sum_k a[c][k][i] b[c][k][j]
 *   a, b        device bf16 [c_h][B][ld] (ld >= B, a multiple of 8);
 *   x           device float32 [c_h][B][ldx], ldx >= B and a multiple of 4; columns < B are written;
 *   accumulate  0: x is overwritten; 1: the product is added to x (TMA reduce-add: each sum is formed and
 *               rounded to float32 where it lands). The blocks of a split grid's k axis are added one
 *               after another into the same x. */
tm_status tm_contract_block(tm_ctx* ctx, const void* a, const void* b, int B, int ld, tm_direction dir,
                            float* x, int ldx, int accumulate, void* stream);

/* Gradients of the layer's parameters: device float32 arrays, each shaped as
 * the tm_weights member of the same name. A NULL member is not written. */
typedef struct {
  float *ln_in_gamma, *ln_in_beta;
  float *w_a, *w_ga, *w_b, *w_gb;
  float *w_g;
  float *ln_out_gamma, *ln_out_beta;
  float *w_o;
} tm_grads;

/* Backward pass of one update, for training (the pages call fine-tuning at
 * larger crops essential: section "A pegadinha" of the BioNeMo context-
 * parallelism page named above). For the cotangent dout of out = update(z)
 * (the gradient of a scalar loss L with respect to out) it writes
 *   dz    = dL/dz   = J_z^T dout,   and
 *   grads = dL/dW for every parameter (overwritten, not accumulated),
 * with the chain rule taken through the definition in the header comment:
 *   dy = dout*g, dgg = dout*y*g(1-g) (g = sigmoid(W_g zh), y = W_o LN_out(x));
 *   LayerNorm backward over c_h gives dx;
 *   outgoing: da = dX b, db = dX^T a  /  incoming: da = b dX^T, db = a dX
 *     (per channel, over the N x N planes);
 *   the gate backward of a and b (masked like a and b) and W^T products give
 *   dzh; LayerNorm backward over c_z gives dz.
 * It recomputes a, b and x from z (no state is kept from a forward call).
 *   z      device [N][N][c_z] of dtype;
 *   mask   device float32 [N] or NULL, as for tm_forward;
 *   dout   device [N][N][c_z] of dtype;
 *   dz     device [N][N][c_z] of dtype; may be dout itself (dout is fully read
 *          before dz is written), must not otherwise overlap dout or z;
 *   grads  device pointers (float32), or NULL to skip every parameter gradient.
 * Precisions: TM_F32 keeps every intermediate in float32 on the CUDA cores.
 * TM_BF16 recomputes a and b as the forward stores them (bf16 values, held as
 * fp16 times powers of two) and x in float32; dL/dx leaves the output backward
 * as fp16 under a power of two fixed by a bound on it (a constant of the weights
 * times the largest |dout|), and its contractions with b and a, the per-pair
 * W^T products and the parameter sums over the N^2 pairs run on the tensor
 * cores from fp16 operands with float32 accumulation; dA and dB are float32.
 * Schedule and workspace for TM_BF16: a, b and dX (fp16 planes, 768 B per pair)
 * plus, per row block of B rows, dA, dB and the gate's part of dL/dzh in float32
 * and one B x B block of x: about 2.3 kB per pair for the whole grid at once
 * (30 GB at N = 3605, 98 GB at N = 6500); when that would pass 100 GiB (or the
 * workspace limit), the grid goes in blocks of B (2560, 2048, 1536, ...; N =
 * 10000: B = 1536, 103 GB): x and the output backward block by block for dX,
 * then row block by row block x again for dL/dzh, dA and dB of the rows and the
 * projection backward over them. The result does not depend on B (dz bit for
 * bit; the parameter sums up to float32 reordering). opt->block sets B (>= 128
 * and a multiple of 8, or >= N for the whole grid; bf16 only). Beyond the
 * workspace limit it returns TM_ERR_OOM before any launch. opt: timeout_ms,
 * workspace_limit and block apply; x_storage and residual must be 0.
 * Stream-ordered like tm_forward. */
tm_status tm_backward(tm_ctx* ctx, const void* z, const float* mask, int N, tm_dtype dtype,
                      tm_direction dir, const void* dout, void* dz, const tm_grads* grads,
                      void* stream, const tm_options* opt);

/* ------------------------------------------------------------------ triangle attention
 * The other O(N^3) operation of the pair stack: the BioIR page ("BioIR da Nvidia
 * acelera previsão de proteínas em 2,9x com PyTorch puro") names triangle
 * operations and pairwise attention among the Pairformer parts its kernels
 * target, without their arithmetic. libtm computes the AlphaFold3/Boltz
 * triangle attention over z [N][N][c_z] with H heads of dimension c:
 *
 *   zh = LayerNorm(z);  q, k, v = W_q zh, W_k zh, W_v zh;  g = sigmoid(W_g zh)
 *   b_jk^h = (W_b zh_jk)^h                                        (pair bias)
 *   starting node: o_ij^h = g_ij^h * sum_k softmax_k(q_ij^h.k_ik^h/sqrt(c) + b_jk^h) v_ik^h
 *                  over keys k with m_i m_k = 1
 *   ending node:   the same on the transposed grid (keys k_kj, v_kj, bias b_ki)
 *   out_ij = W_o [o_ij^1 .. o_ij^H]
 *
 * Linear layers have no bias; a query row with no valid key (a masked token's
 * row for the starting node, column for the ending node) gives o = 0.
 * Supported: bf16 z and out, c_z = 128, H = 4, c = 32. Every intermediate (zh,
 * the weight images, q, k, v, g, the bias b and the softmax weights P, the
 * gated output o) is fp16, zh, v, o and the weight images times powers of two
 * that the weights' bounds fix, as operands of tcgen05 products with float32
 * accumulation; the softmax runs in float32 in base 2, online over key blocks
 * of 64 against a lazy running reference. Weights whose bound on q, k or b
 * reaches 2^15 are refused by tm_attn_create (TM_ERR_UNSUPPORTED). */
typedef enum { TM_ATTN_STARTING = 0, TM_ATTN_ENDING = 1 } tm_attn_node;

/* Host float32 arrays, Linear layout [out][in]. */
typedef struct {
  const float *ln_gamma, *ln_beta;         /* [c_z]         */
  const float *w_q, *w_k, *w_v, *w_g;      /* [H c][c_z]    */
  const float *w_b;                        /* [H][c_z]      */
  const float *w_o;                        /* [c_z][H c]    */
} tm_attn_weights;

/* A context holding one triangle attention layer (freed by tm_destroy; the
 * update's calls reject it with TM_ERR_INVALID). Returns TM_ERR_INVALID for a
 * NULL argument, TM_ERR_UNSUPPORTED for any shape but c_z = 128, H = 4,
 * c = 32 or for weights that could push q, k or the bias past fp16's range.
 * Synchronous; the caller may free its arrays afterwards. */
tm_status tm_attn_create(int c_z, int heads, int c_head, const tm_attn_weights* w, tm_ctx** out_ctx);

/* out = triangle attention of the given node over z.
 *   z     device bf16 [N][N][c_z]; mask device float32 [N] or NULL;
 *   out   device bf16 [N][N][c_z], must not overlap z.
 * Workspace: about 1.3 kB per pair (q, k, v, g, o and the bias, fp16).
 * opt: timeout_ms and workspace_limit apply, other fields must be 0. dtype
 * TM_F32 returns TM_ERR_UNSUPPORTED. Stream-ordered like tm_forward. */
tm_status tm_attn_forward(tm_ctx* ctx, const void* z, const float* mask, int N, tm_dtype dtype,
                          tm_attn_node node, void* out, void* stream, const tm_options* opt);

/* Synchronise `stream` and return the device status word (TM_OK or
 * TM_ERR_TIMEOUT), clearing it. */
tm_status tm_sync_status(tm_ctx* ctx, void* stream);

/* Per-kernel timing with CUDA events recorded on the launch stream.
 * enable != 0 starts recording (and clears the totals). */
typedef struct {
  int launches[12];    /* projection, contraction, finish, float32 kernels,
                          output backward, projection backward, other
                          backward kernels (transpose, sums), unused,
                          attention projection, attention, attention
                          output, unused                                    */
  double ms[12];       /* summed event-measured durations                  */
  long long units[12]; /* pairs processed (projection, finish, backward,
                          attention) or channel x output-pair products
                          (contraction)                                     */
} tm_timing;
tm_status tm_set_timing(tm_ctx* ctx, int enable);
/* Synchronises the recorded events and fills *t. */
tm_status tm_get_timing(tm_ctx* ctx, tm_timing* t);

/* Number of kernel launches made by this ctx since creation. */
long long tm_launch_count(const tm_ctx* ctx);

/* Bytes of workspace currently held by the ctx. */
size_t tm_workspace_bytes(const tm_ctx* ctx);

/* The shape a ctx was created with: *c_z, *c_hidden, and *layer = 0 for a
 * triangle multiplicative update (tm_create), 1 for triangle attention
 * (tm_attn_create; c_hidden is then heads * c_head). NULL outputs are skipped.
 * TM_ERR_INVALID for a NULL ctx. Lets a binding check tensor shapes before it
 * hands pointers to a call that cannot see the buffers' sizes. */
tm_status tm_ctx_info(const tm_ctx* ctx, int* c_z, int* c_hidden, int* layer);

/* Watchdog self-test: launches one small kernel whose wait on an mbarrier
 * that nothing arrives at runs out after timeout_ms (1..10000) and records
 * TM_ERR_TIMEOUT in the ctx's status word, then returns. The call itself
 * returns TM_OK once launched; a following tm_sync_status returns
 * TM_ERR_TIMEOUT, and the ctx stays usable. Exercises the same bounded wait
 * every libtm kernel uses, without faulting or hanging the GPU. */
tm_status tm_watchdog_selftest(tm_ctx* ctx, int timeout_ms, void* stream);

/* Probe of the special-function pipe: the rate of ex2.approx.ftz.f32 (the
 * exponential of the triangle attention's softmax) on this device, from a
 * kernel of independent exponential chains on every SM (4 CTAs of 512 threads
 * per SM, 8 x 20000 exponentials per thread), timed with CUDA events on
 * `stream`. Blocks the calling thread until the probe has run. *per_second:
 * exponentials per second over the whole device. For rooflines; launches no
 * library work. Errors: TM_ERR_INVALID (NULL argument), TM_ERR_CUDA. */
tm_status tm_probe_ex2_rate(tm_ctx* ctx, double* per_second, void* stream);

/* Allocation-free forward (the pages have no counterpart; this is a service of
 * the library). Same contract and result as tm_forward for TM_BF16 and
 * 1 <= N <= 128, for callers that may not allocate device memory: code whose
 * device memory all belongs to another allocator or to a fixed budget, and code
 * that must not pay a device allocation's host-side stall. The a, b and x
 * scratch lives in one static 12.1 MiB device array inside libtm, which every
 * GPU that loads the library holds until the process exits; the call itself
 * allocates nothing. The first call on a device looks up that array's device
 * address (once per device, with the device current), so make that first call
 * before any stream capture. N > 128 returns TM_ERR_UNSUPPORTED. All calls
 * share the one array: calls whose work overlaps on the GPU (other streams,
 * other host threads, other contexts on the same device) race on it and must be
 * serialised by the caller. The timing of tm_set_timing does not cover it. */
tm_status tm_forward_noalloc(tm_ctx* ctx, const void* z, const float* mask, int N, tm_direction dir,
                             void* out, void* stream);

/* Static text of a status code; never NULL. */
const char* tm_status_string(tm_status s);

/* Detail of the ctx's last error ("" if none); valid until the next call. */
const char* tm_last_error(const tm_ctx* ctx);

/* Free the workspace and weights (after synchronising the device). NULL is a no-op. */
void tm_destroy(tm_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* TM_H */
