// Internal launchers shared by the translation units of libgemma3attn.so.
// Nothing here is part of the C ABI (see include/gemma3_attn.h).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace g3 {

enum DType : int { kBF16 = 0, kF16 = 1, kF32 = 2 };

// cuTensorMapEncodeTiled, fetched from the driver at first use (the library
// does not link libcuda, so it loads on machines without a driver).
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

int num_sms();

// Raises `kern`'s dynamic shared-memory limit to `smem_bytes` on the current
// device, once per (kernel, device) and safe to call from several host
// threads; `regs`, if given, receives the kernel's registers per thread.
cudaError_t prepare_kernel(const void* kern, int smem_bytes, int* regs = nullptr);

// Launch `kern` on `stream` with programmatic dependent launch allowed: the
// grid may start while the previous kernel on the stream is finishing, and
// its pdl_enter() (ptx.cuh) waits for that kernel before any global-memory
// access.  Only kernels that begin with pdl_enter() are launched this way.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// The same launch in thread-block clusters of cluster_x CTAs along x
// (grid.x a multiple of cluster_x).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               int cluster_x, cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Rows per tile of the tcgen05 GEMM for later launches: 0 (chosen per
// launch), 128 or 256; returns the previous value, or -1 for another value.
int set_gemm_tile_rows(int rows);

// C[M,N] = A[M,K] * W[N,K]^T, operands in in_dtype (bf16|f16), fp32
// accumulation, C in out_dtype.  M <= kSkinnyMaxRows goes to
// launch_linear_skinny, everything else to the tcgen05 GEMM.
// With pad_lens, M = B * seg_T rows of B segments with trailing padding
// (seg_T a multiple of 128): the 128-row tiles holding only pad rows are not
// computed, and their rows of C are written as zeros when zero_pad_tiles,
// else left unwritten.
cudaError_t launch_linear(const void* A, long lda, const void* W, long ldw, void* C, long ldc,
                          int M, int N, int K, int in_dtype, int out_dtype, cudaStream_t stream,
                          int* status, int max_ctas, const int32_t* pad_lens = nullptr,
                          int seg_T = 0, bool zero_pad_tiles = false);

// The same product for M <= kSkinnyMaxRows (bound by reading W from HBM):
// W streamed by TMA into the 128-row side of the tcgen05 MMA, K split over
// a cluster; K % 8 == 0, 16-byte aligned rows.  Its bounded waits record
// into `status`.
constexpr int kSkinnyMaxRows = 16;
cudaError_t launch_linear_skinny(const void* A, long lda, const void* W, long ldw, void* C,
                                 long ldc, int M, int N, int K, int in_dtype, int out_dtype,
                                 cudaStream_t stream, int* status);
// Two such products of the same A in one launch: C1 = A W1^T (N1 columns,
// a multiple of 128) and C2 = A W2^T (N2 columns).
cudaError_t launch_linear_skinny2(const void* A, long lda, const void* W1, long ldw1, void* C1,
                                  long ldc1, int N1, const void* W2, long ldw2, void* C2,
                                  long ldc2, int N2, int M, int K, int in_dtype, int out_dtype,
                                  cudaStream_t stream, int* status);

// Z[M, D_ff] (fp16) = GELU_tanh(A Wg^T) * (A Wu^T), Wgu = [Wg; Wu] of shape
// [2*D_ff, K] (the transposed gating weight (2, D_ff, D) viewed as rows).
cudaError_t launch_geglu(const void* A, long lda, const void* Wgu, long ldw, void* Z, long ldz,
                         int M, int D_ff, int K, int in_dtype, cudaStream_t stream, int* status);

// C[M, N] (fp16) = A W^T with the attention prologue in the epilogue: columns
// [0, n_norm) are head vectors of d_h that get RMSNorm with (1 + gamma), RoPE
// at pos[row] with (rope_base, rope_scale) and the factor `scale`; the other
// columns are stored as they are.  Requires linear_qknorm_fusable().
bool linear_qknorm_fusable(int M, int N, int n_norm, int d_h);
cudaError_t launch_linear_qknorm(const void* A, long lda, const void* W, long ldw, void* C,
                                 long ldc, int M, int N, int K, int in_dtype, const void* gamma,
                                 const int32_t* pos, int d_h, int n_norm, double rope_base,
                                 double rope_scale, float scale, cudaStream_t stream,
                                 int* status);

// The Q and KV projections with that epilogue in one launch: Qout [M, HD]
// (all head vectors, gamma_q, query_scale) and KVout [M, 2*KVD] (K' head
// vectors with gamma_k, then V as it is), Wq [HD, K] and Wkv [2*KVD, K]
// sharing the row stride ldw.
cudaError_t launch_qkv_qknorm(const void* A, long lda, const void* Wq, const void* Wkv, long ldw,
                              void* Qout, long ldq, void* KVout, long ldkv, int M, int HD, int KVD,
                              int K, int in_dtype, const void* gamma_q, const void* gamma_k,
                              const int32_t* pos, int d_h, double rope_base, double rope_scale,
                              float query_scale, cudaStream_t stream, int* status,
                              const int32_t* pad_lens = nullptr, int seg_T = 0);

// Where a decode step's new K'/V rows also go: row m = b*T + t to slot
// b*S + end + t of the fp16 caches Kc / Vc ([B, S, H_kv*d_h]), its position
// pos[m] (or -1 for t past the valid length T - pad_lens[b]) to posc
// ([B, S]); V is read from rows of V with stride ldv.  Kc == nullptr: none.
struct CacheRows {
  void* Kc = nullptr;
  void* Vc = nullptr;
  int32_t* posc = nullptr;
  const void* V = nullptr;
  long ldv = 0;
  const int32_t* pad_lens = nullptr;
  int T = 1, S = 0, end = 0;
  // With span_part on a local layer (window > 0): the launch also writes the
  // visible span of each row ([B, nchunk], nchunk = cached_span_chunks) for
  // the cache attention that follows (launch_cached_attention with prepared).
  int32_t* span_part = nullptr;
  int window = 0, nchunk = 0;
};

// In place on fp16 rows: Q[m, h*d_h:(h+1)*d_h] and K[m, j*d_h:(j+1)*d_h] get
// last-axis RMSNorm, (1 + gamma), RoPE; Q also the query scale.  With
// cache.Kc the normalised K' rows, the V rows and the positions are also
// written to their cache slots (the cache write of a decode step).
cudaError_t launch_qk_norm_rope(void* Q, long ldq, void* K, long ldk, const void* gamma_q,
                                const void* gamma_k, const int32_t* pos, int M, int H, int H_kv,
                                int d_h, double rope_base, double rope_scale, float query_scale,
                                cudaStream_t stream, const CacheRows& cache = CacheRows{});

// Flash attention forward over Q' [B,T,H,d_h] fp16 and K'/V rows of an fp16
// buffer with row stride ldkv (K' at column j*d_h, V at column v_off + j*d_h).
// Writes O [B,T,H,d_h] in o_dtype (bf16|f16; may alias Q'); rows past the
// valid length are 0.  sched: kAttnSchedBytes of device scratch for the
// dynamic work order, or null for the static order; its counter is zeroed
// here before the launch unless sched_zeroed says the caller already zeroed
// it on the stream (a pipeline does so at its start, so that no memset
// separates the kernels before and after the attention).
constexpr size_t kAttnSchedBytes = 256;
cudaError_t launch_flash_attention(const void* Q, const void* K, const void* V, long ldkv,
                                   void* O, int o_dtype, const int32_t* pad_lens, int B, int T,
                                   int H, int H_kv, int d_h, int window, void* sched,
                                   cudaStream_t stream, int* status, bool sched_zeroed = false);
// The d_h = 128 kernel behind launch_flash_attention (two query tiles per
// CTA); same arguments, G = H / H_kv in {1, 2, 4}.
cudaError_t launch_flash_attention_pair(const void* Q, const void* K, const void* V, long ldkv,
                                        void* O, int o_dtype, const int32_t* pad_lens, int B,
                                        int T, int H, int H_kv, int window, void* sched,
                                        cudaStream_t stream, int* status, bool sched_zeroed);

// Rows of M = B * seg_T in B segments of seg_T rows, segment b's last
// pad_lens[b] rows padding (pad_lens null: no padding information).
struct PadRows {
  const int32_t* pad_lens = nullptr;
  int seg_T = 0;
};

// u[m,:] = RMSNorm(x[m,:]) * (1 + gamma) over D, x in x_dtype (bf16|f32), u in
// u_dtype (bf16|f16).  With `pad`, rows in 128-row tiles of pad rows alone
// (seg_T a multiple of 128: the tiles the projections skip) are not written.
cudaError_t launch_rmsnorm_rows(const void* x, int x_dtype, const void* gamma, void* u,
                                int u_dtype, int M, int D, cudaStream_t stream,
                                const PadRows& pad = {});

// dst[i] = src[i] converted bf16 -> f16 (round to nearest even), n elements.
cudaError_t launch_cast_bf16_f16(const void* src, void* dst, size_t n, cudaStream_t stream);

// x[m, :] = E[tokens[m], :] * scale (fp32), E [V, D] bf16; bad token ids give
// a zero row and a device status error.
cudaError_t launch_embed_rows(const int32_t* tokens, const void* E, int V, int D, int M,
                              float scale, float* x, cudaStream_t stream, int* status);

// y[m,:] = x[m,:] + RMSNorm(a[m,:]) * (1 + gamma); a f32, x bf16|f32, y f32.
// With `pad`, pad rows (whose a is zero, an attention layer's output there)
// get y = x without reading a, and are left alone when y is x.
cudaError_t launch_postnorm_residual(const float* a, const void* x, int x_dtype,
                                     const void* gamma, float* y, int M, int D,
                                     cudaStream_t stream, const PadRows& pad = {});

// KV cache: copy the T new tokens' K' and V rows (KVD = H_kv*d_h fp16 each,
// row (b, t) at K_rows/V_rows + (b*T + t)*ld) into slot end + t of the caches
// [B, S, KVD] and store their positions (-1 for pad tokens) in pos_cache [B, S].
cudaError_t launch_kv_cache_append(const void* K_rows, const void* V_rows, long ld,
                                   const int32_t* segment_pos, const int32_t* pad_lens, int B,
                                   int T, int S, int end, int KVD, void* K_cache, void* V_cache,
                                   int32_t* pos_cache, cudaStream_t stream);

// Workspace of launch_cached_attention (depends only on the shapes and S).
size_t cached_attention_ws_bytes(int B, int T, int S, int H, int H_kv, int d_h);

// Attention of T query tokens per row (written to slots end..end+T-1) over a
// left-aligned K'/V cache [B, S, H_kv, d_h] fp16 with stored positions
// pos_cache [B, S]; Q' and O [B, T, H, d_h] (O in o_dtype, may alias Q').
// prepared: the kernel before it on the stream already wrote the local
// layer's span (CacheRows with span_part); otherwise this call scans it first.
cudaError_t launch_cached_attention(const void* Q, const void* K_cache, const void* V_cache,
                                    const int32_t* pos_cache, const int32_t* qpos,
                                    const int32_t* pad_lens, void* O, int o_dtype, int B, int T,
                                    int S, int end, int H, int H_kv, int d_h, int window,
                                    void* ws, cudaStream_t stream, int* status,
                                    bool prepared = false);

// Where launch_cached_attention keeps its span and split partials in a
// workspace `ws` (bytes: the total), and the span chunks of a call.
struct CachedAttnLayout {
  int32_t* span_part;
  float* part;
  int nchunk;
  size_t bytes;
};
CachedAttnLayout cached_attention_layout(void* ws, int B, int T, int S, int H, int H_kv, int d_h);
int cached_span_chunks(int T, int end);

}  // namespace g3
