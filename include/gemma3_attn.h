/*
 * gemma3_attn.h -- C ABI of libgemma3attn.so: the forward pass of the Gemma 3
 * attention block on one NVIDIA GB300 (sm_103a).
 *
 * What it computes is defined by four pages, cited below by title and section:
 *   [AB] "Gemma 3 Attention Block"        Overview; How it works (Projections,
 *        QK-norm then RoPE then scale, Scores, Routing)
 *   [FB] "Full Gemma 3 Block"             How it works (Block.__call__ equations)
 *   [RT] "Global vs Local Layer Routing"  How it works; Watch-outs
 *   [QK] "QK-Norm"                        How it works (RMSNorm equation); Watch-outs
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers, 16-byte aligned, row-major and
 *     contiguous unless a leading dimension is given.  bf16 / f16 tensors are
 *     passed as void* and hold IEEE binary16 / bfloat16 bit patterns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *     asynchronous on that stream and never synchronises; read results after
 *     synchronising the stream yourself.
 *   - The caller owns every buffer.  The library never allocates device memory;
 *     scratch space is the caller's `workspace` (see gemma3_attn_workspace_size),
 *     or, for gemma3_attn_forward_noalloc only, a fixed array inside the library.
 *     Inputs are read only; only `out`/`y` and `workspace` are written.
 *   - Every function returns a status (GEMMA3_OK = 0 or a negative error) and
 *     validates all arguments before launching anything.  Kernels that lose a
 *     synchronisation event stop after a bounded wait and record an error that
 *     gemma3_attn_check_status() reports; they never hang or trap.
 *   - Calls on different streams need distinct workspaces.
 */
#ifndef GEMMA3_ATTN_H_
#define GEMMA3_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum {
  GEMMA3_OK = 0,
  GEMMA3_ERR_INVALID_ARG = -1, /* null pointer, bad shape or out-of-range value */
  GEMMA3_ERR_MISALIGNED = -2,  /* pointer or row stride not 16-byte aligned */
  GEMMA3_ERR_UNSUPPORTED = -3, /* d_h not in {128, 256}, G not in {1, 2, 4}, not sm_103 */
  GEMMA3_ERR_CUDA = -4,        /* a CUDA runtime call or kernel launch failed */
  GEMMA3_ERR_TIMEOUT = -5,     /* a kernel gave up on a bounded wait (device status word) */
  GEMMA3_ERR_WORKSPACE = -6,   /* workspace smaller than gemma3_*_workspace_size() */
  GEMMA3_ERR_BAD_INPUT = -7    /* a kernel found invalid data (a token id outside [0, V)) */
};

/* Attention types of [RT] How it works (AttentionType enum). */
enum { GEMMA3_LOCAL_SLIDING = 0, GEMMA3_GLOBAL = 1 };

/* Element types for the stage entry points. */
enum { GEMMA3_BF16 = 0, GEMMA3_F16 = 1, GEMMA3_F32 = 2 };

/* Released sizes named by the pages ([AB] Overview, [RT] How it works). */
enum { GEMMA3_270M = 0, GEMMA3_1B = 1, GEMMA3_4B = 2, GEMMA3_12B = 3, GEMMA3_27B = 4 };

/* Layer shape: batch B, sequence T, model width D, H query heads, H_kv
 * key/value heads (H % H_kv == 0, G = H / H_kv), head dim d_h. */
typedef struct {
  int B, T, D, H, H_kv, d_h;
} gemma3_attn_dims;

/* ------------------------------------------------------------------ routing */

/* Attention type of layer `layer` (0-based) in a stack of `num_layers`:
 * P[layer mod 6] with P = (L,L,L,L,L,G); a depth that is not a multiple of 6
 * ends with the prefix P[:N % 6], so leftover layers are local ([RT] How it
 * works, Watch-outs).  Returns GEMMA3_LOCAL_SLIDING or GEMMA3_GLOBAL, or
 * GEMMA3_ERR_INVALID_ARG when layer is not in [0, num_layers). */
int gemma3_layer_attn_type(int layer, int num_layers);

/* Per-layer hyper-parameters that the type selects ([RT] How it works,
 * Transformer.setup mapping; [AB] Overview): local layers RoPE base 1e4,
 * scale 1, window 1024 (512 on 270M/1B); global layers base 1e6, scale 8 on
 * 4B/12B/27B and 1 on 270M/1B, window 0 (= none).  Any output pointer may be
 * NULL.  Returns the attention type or a negative status. */
int gemma3_layer_config(int layer, int num_layers, int model_size, int* attn_type, int* window,
                        double* rope_base, double* rope_scale);

/* query_pre_attn_scalar ([AB] How it works, query scale): d_h^-1/2, or
 * (D/H)^-1/2 on 27B.  Writes it to *alpha; returns a status. */
int gemma3_query_scale(int model_size, int D, int H, int d_h, float* alpha);

/* ------------------------------------------------------------ one attention layer */

/* Bytes of workspace gemma3_attn_forward needs for `dims` (written to *bytes):
 * Q/O rows [B*T, H*d_h] and K/V rows [B*T, 2*H_kv*d_h], 2 bytes per element. */
int gemma3_attn_workspace_size(const gemma3_attn_dims* dims, size_t* bytes);

/* Forward pass of one Gemma 3 attention layer ([AB] How it works, steps in
 * order):
 *   Q = x Wq^T, [K|V] = x Wkv^T                     (Projections; fp32 accumulate)
 *   Q, K <- RMSNorm over d_h * (1 + gamma_q|gamma_k), eps 1e-6   ([QK])
 *   Q, K <- RoPE(rope_base, rope_scale) at segment_pos; Q <- query_scale * Q
 *   logits = Q K^T per head, kv head h / G; keep s <= t, s < T - pad_b and,
 *   for GEMMA3_LOCAL_SLIDING, s > t - window; softmax over s; O = P V
 *   out = O Wo^T                                    (attn_vec_einsum)
 * Arguments:
 *   x            [B, T, D] bf16
 *   segment_pos  [B, T] int32 RoPE positions (0 <= pos < 2^24)
 *   pad_lens     [B] int32 trailing pad count per batch row (0 <= pad_b <= T),
 *                or NULL for none.  Rows t >= T - pad_b of `out` are written 0.
 *   Wq           [H*d_h, D] bf16, row n = h*d_h + c
 *   Wkv          [2, H_kv*d_h, D] bf16, [0] = K, [1] = V
 *   Wo           [D, H*d_h] bf16
 *   gamma_q/k    [d_h] bf16 each (separate scales, shared across heads)
 *   attn_type    GEMMA3_LOCAL_SLIDING (window >= 1) or GEMMA3_GLOBAL (window ignored)
 *   rope_base, rope_scale  > 0;  query_scale  the query scale alpha
 *   out          [B, T, D] bf16
 *   workspace    >= gemma3_attn_workspace_size() bytes, 256-byte aligned
 * Limits: d_h in {128, 256}; G in {1, 2, 4}; D % 8 == 0; B*T < 2^31. */
int gemma3_attn_forward(const gemma3_attn_dims* dims, const void* x, const int32_t* segment_pos,
                        const int32_t* pad_lens, const void* Wq, const void* Wkv, const void* Wo,
                        const void* gamma_q, const void* gamma_k, int attn_type, int window,
                        double rope_base, double rope_scale, float query_scale, void* out,
                        void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------- one attention layer, no allocation */

/* The pages have no counterpart to this entry point; it exists for callers
 * that cannot give the library a workspace, e.g. code that may not call
 * cudaMalloc (a latency-critical loop, a process whose device memory is owned
 * by another framework's pool, an interface that only carries input and
 * output buffers).
 *
 * Same computation, arguments and output as gemma3_attn_forward, but the
 * intermediate rows live in a fixed scratch array inside the library
 * (gemma3_attn_noalloc_max_scratch() bytes = 16 MiB per device, reserved on
 * every GPU that loads the library until the process exits).  The call makes
 * no device allocation of any kind.
 *   - Problems whose workspace (gemma3_attn_workspace_size) exceeds the
 *     scratch size are refused with GEMMA3_ERR_WORKSPACE before any launch.
 *   - The first call on each device looks up the scratch array's device
 *     address (cudaGetSymbolAddress, no allocation); make that first call
 *     before capturing a stream on that device.
 *   - All calls share the one array and nothing in it needs clearing between
 *     calls; calls whose kernels overlap on the GPU (different streams, or
 *     unordered host threads) race on it: serialise them. */
int gemma3_attn_forward_noalloc(const gemma3_attn_dims* dims, const void* x,
                                const int32_t* segment_pos, const int32_t* pad_lens,
                                const void* Wq, const void* Wkv, const void* Wo,
                                const void* gamma_q, const void* gamma_k, int attn_type,
                                int window, double rope_base, double rope_scale,
                                float query_scale, void* out, void* stream);

/* Size in bytes of the scratch array gemma3_attn_forward_noalloc uses. */
size_t gemma3_attn_noalloc_max_scratch(void);

/* ------------------------------------------------------- one block-attention layer */

/* Workspace of gemma3_block_attn_forward: that of gemma3_attn_forward, fp16
 * copies of Wq, Wkv and Wo, [B*T, D] fp16 (normed input) and [B*T, D] fp32
 * (attention output). */
int gemma3_block_attn_workspace_size(const gemma3_attn_dims* dims, size_t* bytes);

/* Attention half of a Gemma 3 block ([FB] How it works, first three lines):
 *   a = Attn(RMSNorm_pre(x));  a <- RMSNorm_post(a);  y = x + a
 * with D-axis RMSNorms, eps 1e-6, (1 + gamma).  x is [B, T, D] in x_dtype
 * (GEMMA3_BF16 or GEMMA3_F32); y is [B, T, D] fp32 and may alias x when
 * x_dtype is GEMMA3_F32.  gamma_pre / gamma_post are [D] bf16; the other
 * arguments are those of gemma3_attn_forward.  Pad rows get a = 0, so y = x.
 * Precision: the normed input and the attention output are kept in fp16
 * (the bf16 weights are cast to fp16 copies in the workspace), since in a
 * stack of layers bf16 rounding of those activations accumulates past the
 * tolerance of the block output; the residual stream stays fp32. */
int gemma3_block_attn_forward(const gemma3_attn_dims* dims, const void* x, int x_dtype,
                              float* y, const int32_t* segment_pos, const int32_t* pad_lens,
                              const void* Wq, const void* Wkv, const void* Wo,
                              const void* gamma_q, const void* gamma_k, const void* gamma_pre,
                              const void* gamma_post, int attn_type, int window,
                              double rope_base, double rope_scale, float query_scale,
                              void* workspace, size_t workspace_bytes, void* stream);

/* ----------------------------------------------------- feed-forward half, full block */

/* Workspace of gemma3_block_ffn_forward for M = B*T rows: [M, D] fp16 normed
 * input, [M, D_ff] fp16 gated activations, [M, D] fp32 FFN output and fp16
 * copies of the two weights. */
int gemma3_block_ffn_workspace_size(int M, int D, int D_ff, size_t* bytes);

/* Feed-forward half of a Gemma 3 block ([FB] How it works, last three lines
 * of Block.__call__ and the MLP paragraph):
 *   m = FFN(RMSNorm_pre-ffn(h));  m <- RMSNorm_post-ffn(m);  y = h + m
 *   FFN(u) = (GELU(u Wg^T) * (u Wu^T)) Wd^T, GELU in its tanh form.
 * Arguments:
 *   h, y         [M, D] fp32 (y may alias h); D % 8 == 0, D_ff % 8 == 0
 *   gamma_*_ffn  [D] bf16, (1 + gamma) RMSNorms with eps 1e-6
 *   W_gating     [2, D_ff, D] bf16, the page's transposed gating weight:
 *                [0] = W_g (gate, takes the GELU), [1] = W_u (up)
 *   W_down       [D, D_ff] bf16: the page's (D_ff, D) linear stored
 *                transposed (K-major, like every weight of this library)
 * The normed input and the gated activations are fp16 (the weights are cast
 * to fp16 copies in the workspace), as in gemma3_block_attn_forward.  Rows
 * are independent; pad rows are computed like any other. */
int gemma3_block_ffn_forward(int M, int D, int D_ff, const float* h, float* y,
                             const void* gamma_pre_ffn, const void* gamma_post_ffn,
                             const void* W_gating, const void* W_down, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Workspace of gemma3_block_forward: the larger of its two halves'. */
int gemma3_block_workspace_size(const gemma3_attn_dims* dims, int D_ff, size_t* bytes);

/* The whole Gemma 3 block ([FB] How it works, Block.__call__): the
 * block-attention sandwich of gemma3_block_attn_forward, then the
 * feed-forward sandwich of gemma3_block_ffn_forward.  x [B, T, D] bf16 or
 * fp32 (x_dtype), y [B, T, D] fp32 (may alias an fp32 x); the other
 * arguments are those two calls'. */
int gemma3_block_forward(const gemma3_attn_dims* dims, int D_ff, const void* x, int x_dtype,
                         float* y, const int32_t* segment_pos, const int32_t* pad_lens,
                         const void* Wq, const void* Wkv, const void* Wo, const void* gamma_q,
                         const void* gamma_k, const void* gamma_pre_attn,
                         const void* gamma_post_attn, const void* gamma_pre_ffn,
                         const void* gamma_post_ffn, const void* W_gating, const void* W_down,
                         int attn_type, int window, double rope_base, double rope_scale,
                         float query_scale, void* workspace, size_t workspace_bytes,
                         void* stream);

/* ------------------------------------------------------------------ the model */

/* Device pointers of one block's weights (as gemma3_block_forward takes them). */
typedef struct {
  const void* Wq;              /* [H*d_h, D] bf16 */
  const void* Wkv;             /* [2, H_kv*d_h, D] bf16 */
  const void* Wo;              /* [D, H*d_h] bf16 */
  const void* gamma_q;         /* [d_h] bf16 */
  const void* gamma_k;         /* [d_h] bf16 */
  const void* gamma_pre_attn;  /* [D] bf16 */
  const void* gamma_post_attn; /* [D] bf16 */
  const void* gamma_pre_ffn;   /* [D] bf16 */
  const void* gamma_post_ffn;  /* [D] bf16 */
  const void* W_gating;        /* [2, D_ff, D] bf16 */
  const void* W_down;          /* [D, D_ff] bf16 */
} gemma3_block_weights;

/* Workspace of gemma3_model_forward. */
int gemma3_model_workspace_size(const gemma3_attn_dims* dims, int D_ff, int V, size_t* bytes);

/* The model around the blocks ([FB] How it works, last paragraph):
 *   x = E[tokens] * sqrt(D);  x <- Block_l(x) for l = 0..num_layers-1;
 *   logits = RMSNorm_final(x) E^T  (read-out through the embedding table).
 * Block l is gemma3_block_forward with the type, window and RoPE pair that
 * gemma3_layer_config(l, num_layers, model_size) gives and the query scale of
 * gemma3_query_scale(model_size, ...).  tokens [B, T] int32 in [0, V) (others
 * give zero rows and GEMMA3_ERR_BAD_INPUT from gemma3_attn_check_status);
 * E [V, D] bf16; layers: HOST array of num_layers structs of device
 * pointers; gamma_final [D] bf16; logits [B, T, V] fp32 (V % 4 == 0).  The
 * residual stream stays fp32 between blocks; the final norm is rounded to
 * bf16 for the read-out GEMM.  Pad rows run through every block like the
 * other rows (their attention output is 0). */
int gemma3_model_forward(const gemma3_attn_dims* dims, int D_ff, int V, int num_layers,
                         int model_size, const int32_t* tokens, const int32_t* segment_pos,
                         const int32_t* pad_lens, const void* E,
                         const gemma3_block_weights* layers, const void* gamma_final,
                         float* logits, void* workspace, size_t workspace_bytes, void* stream);

/* x[m, :] = E[tokens[m], :] * scale in fp32 ([FB] last paragraph, with
 * scale = sqrt(D)); E [V, D] bf16, D % 8 == 0; x [M, D] fp32. */
int gemma3_embed(const int32_t* tokens, const void* E, int V, int D, int M, float scale, float* x,
                 void* stream);

/* ------------------------------------------------------------------ KV cache */

/* A layer's KV cache ([AB] How it works, Cache): K' (after QK-norm and RoPE)
 * and V of earlier tokens in a left-aligned buffer of S slots per batch row,
 * with the position each slot was written at.
 *   K_cache, V_cache  [B, S, H_kv, d_h] fp16, 16-byte aligned
 *   pos_cache         [B, S] int32; a slot that holds no token stores a
 *                     negative position.  A fresh cache must be all negative
 *                     (cudaMemset to 0xFF gives -1 everywhere).
 * Mask with a cache, for the new token t of row b written to slot end + t
 * (the pages' causal-and-padding mask taken over slots, and the sliding mask
 * evaluated on stored positions, which is why they are stored):
 *   slot s is visible  <=>  s <= end + t  and  pos_cache[b, s] >= 0  and, on a
 *   local layer, segment_pos[b, t] - W < pos_cache[b, s] < segment_pos[b, t] + W.
 * The caller owns the cache and advances end_index itself; nothing wraps. */

/* Workspace of gemma3_attn_forward_cached for T new tokens per row and a
 * cache of S slots. */
int gemma3_attn_cached_workspace_size(const gemma3_attn_dims* dims, int S, size_t* bytes);

/* One attention layer over dims->T new tokens per row with a KV cache.
 * Computes Q, K', V of the new tokens exactly as gemma3_attn_forward, writes
 * K', V and their positions into slots [end_index, end_index + T) of the
 * cache with a dynamic_update_slice (pad tokens, t >= T - pad_lens[b], are
 * stored with position -1), then attends every new token over the cache
 * under the mask above and applies the output projection.
 *   0 <= end_index, end_index + T <= S; segment_pos [B, T] >= 0 for valid
 *   tokens; out [B, T, D] bf16, pad rows 0.  Other arguments as in
 *   gemma3_attn_forward.  T = 1 is one decode step.
 * The attention of few new tokens is bound by reading the cache (HBM); a
 * prompt of >= 128 tokens written at slot 0 of a global layer runs on the
 * tensor-core flash kernel instead, whose mask is the same there. */
int gemma3_attn_forward_cached(const gemma3_attn_dims* dims, int S, int end_index, const void* x,
                               const int32_t* segment_pos, const int32_t* pad_lens,
                               const void* Wq, const void* Wkv, const void* Wo,
                               const void* gamma_q, const void* gamma_k, int attn_type,
                               int window, double rope_base, double rope_scale, float query_scale,
                               void* K_cache, void* V_cache, int32_t* pos_cache, void* out,
                               void* workspace, size_t workspace_bytes, void* stream);

/* The cache write alone: K_rows / V_rows are fp16 rows with stride ld_rows
 * elements, row b*T + t holding token (b, t)'s H_kv*d_h values; they go to
 * slot end_index + t, and pos_cache[b, end_index + t] = segment_pos[b, t]
 * (-1 for pad tokens; pad_lens may be NULL). */
int gemma3_kv_cache_write(const void* K_rows, const void* V_rows, long ld_rows,
                          const int32_t* segment_pos, const int32_t* pad_lens, int B, int T,
                          int S, int end_index, int H_kv, int d_h, void* K_cache, void* V_cache,
                          int32_t* pos_cache, void* stream);

/* Workspace of gemma3_cached_attention. */
int gemma3_cached_attention_workspace_size(int B, int T, int S, int H, int H_kv, int d_h,
                                           size_t* bytes);

/* The attention over a cache alone: Q' [B, T, H, d_h] fp16 (query scale
 * applied) of tokens already written to slots [end_index, end_index + T);
 * O [B, T, H, d_h] in o_dtype (GEMMA3_BF16 | GEMMA3_F16; may alias Q'), pad
 * rows 0; window <= 0 means global.  Mask as above. */
int gemma3_cached_attention(const void* Q, const void* K_cache, const void* V_cache,
                            const int32_t* pos_cache, const int32_t* segment_pos,
                            const int32_t* pad_lens, void* O, int o_dtype, int B, int T, int S,
                            int end_index, int H, int H_kv, int d_h, int window, void* workspace,
                            size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------- stage entry points */

/* C[M, N] = A[M, K] * W[N, K]^T (the projection einsums of [AB] How it
 * works).  A, W in in_dtype (GEMMA3_BF16 | GEMMA3_F16) with row strides lda,
 * ldw (elements); C in out_dtype (GEMMA3_BF16 | GEMMA3_F16 | GEMMA3_F32) with
 * row stride ldc.  fp32 accumulation on the tcgen05 tensor cores.  K % 8 == 0;
 * strides in bytes must be multiples of 16.  max_ctas > 0 caps the
 * persistent grid.  For M <= 16 (a decode step's projections) the product is
 * bound by reading W, and a kernel that streams W once by TMA runs instead:
 * W fills the 128-row side of the tcgen05 MMA, the rows of A its 16-wide
 * side, and the K range of each 128-row tile of W is split over a cluster of
 * up to 8 CTAs whose fp32 partials are summed through distributed shared
 * memory (max_ctas is ignored there).
 * pad_lens NULL: every row is computed.  Else the M rows are M / seg_T
 * segments of seg_T rows (M a multiple of seg_T) of which segment b's last
 * pad_lens[b] are padding: when seg_T is a multiple of 128 (and M > 16),
 * 128-row tiles that hold only pad rows are neither computed nor written
 * (rows an attention layer never reads); every other row is computed as
 * without pad_lens. */
int gemma3_linear(const void* A, long lda, const void* W, long ldw, void* C, long ldc, int M,
                  int N, int K, int in_dtype, int out_dtype, int max_ctas,
                  const int32_t* pad_lens, int seg_T, void* stream);

/* Rows per tile of the tcgen05 projection GEMM for later calls of this
 * process (every entry point whose projections it runs): 0 = chosen per call
 * (the default), 128, or 256.  A 256-row tile is two 128-row halves sharing
 * each staged W tile, applied to plain and GeGLU outputs (outputs with the
 * fused QK-norm/RoPE keep 128 rows); the results are bitwise the same either
 * way, only the speed differs.  Returns the previous setting, or
 * GEMMA3_ERR_INVALID_ARG for any other value.  A process-wide setting: not
 * for threads that want different ones at once. */
int gemma3_set_gemm_tile_rows(int rows);

/* Z[M, D_ff] fp16 = GELU_tanh(A Wg^T) * (A Wu^T), the gating projection of
 * the feed-forward with the GeGLU applied in the GEMM epilogue ([FB] How it
 * works, MLP).  A [M, K] and W_gating [2*D_ff, K] (the (2, D_ff, K) weight
 * viewed as rows: gate rows first) in in_dtype (GEMMA3_BF16 | GEMMA3_F16). */
int gemma3_geglu(const void* A, long lda, const void* W_gating, long ldw, void* Z, long ldz,
                 int M, int D_ff, int K, int in_dtype, void* stream);

/* Q' [M, H*d_h] and [K'|V] [M, 2*H_kv*d_h] (fp16, row strides H*d_h and
 * 2*H_kv*d_h) of M token rows x [M, D] (row stride ldx) in in_dtype: the Q and
 * KV projections ([AB] Projections) with QK-norm, RoPE and the query scale
 * ([QK] How it works; [AB] QK-norm, then RoPE, then scale), exactly the first
 * stage of gemma3_attn_forward.  When H*d_h and H_kv*d_h are multiples of 256
 * and M > 16 this is one GEMM launch whose epilogue normalises and rotates
 * the head vectors from the fp32 accumulator (each tile of x feeds both
 * projections); for M <= 16 (a decode step) the two projections run in one
 * launch of the few-row kernel of gemma3_linear (H*d_h a multiple of 128)
 * followed by gemma3_qk_norm_rope; otherwise the two projections and
 * gemma3_qk_norm_rope.
 * Wq [H*d_h, D], Wkv [2, H_kv*d_h, D] and x in in_dtype; gamma bf16 [d_h].
 * pad_lens / seg_T as in gemma3_linear: in pad-only 128-row tiles of the
 * fused launch the V rows are written as zeros (the attention kernels may
 * read a few of them at a tile edge, weighted by zero) and the Q' and K'
 * rows are left unwritten (no valid query reads them; masked keys' scores
 * are replaced, not weighted). */
int gemma3_qkv_proj_norm_rope(const void* x, long ldx, const void* Wq, const void* Wkv, void* Q,
                              void* KV, int M, int D, int H, int H_kv, int d_h, int in_dtype,
                              const void* gamma_q, const void* gamma_k, const int32_t* pos,
                              double rope_base, double rope_scale, float query_scale,
                              const int32_t* pad_lens, int seg_T, void* stream);

/* C[M, N] fp16 = A W^T with the attention prologue fused into the GEMM
 * epilogue (what gemma3_linear followed by gemma3_qk_norm_rope computes, but
 * from the fp32 accumulator, without the fp16 round trip): columns [0,
 * n_norm) are head vectors of d_h that get RMSNorm with (1 + gamma) ([QK] How
 * it works), RoPE at pos[row] with (rope_base, rope_scale) and the factor
 * `scale` ([AB] QK-norm, then RoPE, then scale); columns from n_norm on are
 * the plain product (the V half of the KV projection).  gamma bf16 [d_h];
 * pos int32 [M].  Requires M > 16, d_h in {128, 256} and n_norm a multiple of
 * 256 with n_norm <= N (else GEMMA3_ERR_UNSUPPORTED); other rules as
 * gemma3_linear.  The layer entry points use it for Q (gamma_q, scale =
 * query_scale, n_norm = N) and for KV (gamma_k, scale 1, n_norm = H_kv*d_h). */
int gemma3_linear_qk_norm_rope(const void* A, long lda, const void* W, long ldw, void* C,
                               long ldc, int M, int N, int K, int in_dtype, const void* gamma,
                               const int32_t* pos, int d_h, int n_norm, double rope_base,
                               double rope_scale, float scale, void* stream);

/* dst[i] = src[i] for i < n, bf16 -> fp16 with round-to-nearest-even
 * (n % 8 == 0; both 16-byte aligned). */
int gemma3_cast_bf16_f16(const void* src, void* dst, size_t n, void* stream);

/* In place on fp16 rows: for every token m and head, RMSNorm over d_h with
 * (1 + gamma_q) (query heads of Q[m, h*d_h : (h+1)*d_h]) or (1 + gamma_k)
 * (key heads of K[m, j*d_h : ...]), then RoPE at position pos[m] with
 * (rope_base, rope_scale), then Q *= query_scale ([QK] How it works: norm,
 * then RoPE, then query scale).  Q [M, ldq], K [M, ldk] fp16; gamma bf16 [d_h]. */
int gemma3_qk_norm_rope(void* Q, long ldq, void* K, long ldk, const void* gamma_q,
                        const void* gamma_k, const int32_t* pos, int M, int H, int H_kv,
                        int d_h, double rope_base, double rope_scale, float query_scale,
                        void* stream);

/* Masked softmax attention ([AB] How it works, Scores): Q' [B, T, H, d_h]
 * fp16 (query scale already applied); K', V rows of fp16 buffers with row
 * stride ldkv elements, head j at column j*d_h ([B*T, ldkv]); O [B, T, H, d_h]
 * in o_dtype (GEMMA3_BF16 | GEMMA3_F16; may alias Q').  Mask and padding as in
 * gemma3_attn_forward (window <= 0 means global / causal only).  scratch: 256
 * bytes of 16-byte-aligned device memory that hold the work counter through
 * which free SMs take the next (heaviest remaining) query tile, or NULL for a
 * fixed assignment; the call zeroes it on `stream` before the launch. */
int gemma3_flash_attention(const void* Q, const void* K, const void* V, long ldkv, void* O,
                           int o_dtype, const int32_t* pad_lens, int B, int T, int H, int H_kv,
                           int d_h, int window, void* scratch, void* stream);

/* u[m, :] = x[m, :] / sqrt(mean(x[m, :]^2) + 1e-6) * (1 + gamma)  ([FB] block
 * norms).  x [M, D] bf16 or fp32 (x_dtype), gamma [D] bf16, u [M, D] in
 * u_dtype (GEMMA3_BF16 | GEMMA3_F16).  pad_lens / seg_T as in gemma3_linear
 * (NULL: every row): rows of 128-row tiles that hold pad rows only (the
 * tiles the projections skip; seg_T a multiple of 128) are not written. */
int gemma3_rmsnorm(const void* x, int x_dtype, const void* gamma, void* u, int u_dtype, int M,
                   int D, const int32_t* pad_lens, int seg_T, void* stream);

/* y = x + RMSNorm(a) * (1 + gamma)  ([FB] post-attention norm + residual).
 * a [M, D] fp32, x [M, D] bf16|fp32, y [M, D] fp32 (may alias an fp32 x).
 * pad_lens / seg_T as in gemma3_linear (NULL: every row): pad rows, where an
 * attention layer's output a is zero, get y = x exactly without a being read
 * (and are not written at all when y is x). */
int gemma3_postnorm_residual(const float* a, const void* x, int x_dtype, const void* gamma,
                             float* y, int M, int D, const int32_t* pad_lens, int seg_T,
                             void* stream);

/* ------------------------------------------------------------------ status */

/* Synchronises `stream`, reads and clears the device status word of the
 * current device.  Returns GEMMA3_OK, GEMMA3_ERR_TIMEOUT (a bounded wait in a
 * kernel expired), GEMMA3_ERR_BAD_INPUT (a kernel found invalid data), or
 * GEMMA3_ERR_CUDA (the stream reported an error). */
int gemma3_attn_check_status(void* stream);

/* Raw device status word of the last check (0 = none; 0x1000 + n = wait site
 * n; 0x2000 = a token id outside [0, V)). */
int gemma3_last_device_status(void);

/* Human-readable text of a status code. */
const char* gemma3_strerror(int status);

/* Runs one kernel whose single wait nothing ever completes, with the given
 * time limit in nanoseconds (1e6 .. 5e9), and returns what
 * gemma3_attn_check_status() reports (GEMMA3_ERR_TIMEOUT when the bounded wait
 * works).  Exercises the failure path without faulting the device. */
int gemma3_selftest_wait_timeout(long long timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMMA3_ATTN_H_ */
