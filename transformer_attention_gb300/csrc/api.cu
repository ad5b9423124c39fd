// C ABI of libgemma3attn.so (declared in include/gemma3_attn.h): argument
// validation, workspace carving, tensor-map creation and launch sequencing on
// the caller's stream.  No entry point allocates device memory.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/gemma3_attn.h"
#include "internal.h"
#include "ptx.cuh"

// Device status word (one per device that loads the library).
__device__ int g3_device_status;

namespace g3 {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
thread_local int t_last_device_status = 0;

int* status_ptr() {
  // The symbol's device address, looked up on the current device each call
  // (cheap; the runtime caches it per context).
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g3_device_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int to_status(cudaError_t e) { return e == cudaSuccess ? GEMMA3_OK : GEMMA3_ERR_CUDA; }

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMMA3_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return GEMMA3_ERR_CUDA;
  if (major != 10 || minor != 3) return GEMMA3_ERR_UNSUPPORTED;
  return GEMMA3_OK;
}

int validate_dims(const gemma3_attn_dims* d) {
  if (d == nullptr) return GEMMA3_ERR_INVALID_ARG;
  if (d->B < 1 || d->T < 1 || d->D < 8 || d->H < 1 || d->H_kv < 1) return GEMMA3_ERR_INVALID_ARG;
  if (d->H % d->H_kv != 0) return GEMMA3_ERR_INVALID_ARG;
  if (d->D % 8 != 0) return GEMMA3_ERR_INVALID_ARG;
  const int G = d->H / d->H_kv;
  if (d->d_h != 128 && d->d_h != 256) return GEMMA3_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4) return GEMMA3_ERR_UNSUPPORTED;
  const long long M = static_cast<long long>(d->B) * d->T;
  if (M >= (1LL << 31)) return GEMMA3_ERR_INVALID_ARG;
  if (static_cast<long long>(d->H) * d->d_h > (1 << 20)) return GEMMA3_ERR_INVALID_ARG;
  return GEMMA3_OK;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct AttnWs {
  size_t q_bytes, kv_bytes, w_bytes, sched_bytes, total;
};

// Workspace of the layer pipeline: Q/O rows, K/V rows and, when the
// activations are fp16, fp16 copies of Wq, Wkv and Wo.
AttnWs attn_ws(const gemma3_attn_dims* d, bool f16_weights = false) {
  const size_t M = static_cast<size_t>(d->B) * d->T;
  AttnWs w;
  w.q_bytes = round_up(M * d->H * d->d_h * 2, 256);
  w.kv_bytes = round_up(M * 2 * d->H_kv * d->d_h * 2, 256);
  const size_t HD = static_cast<size_t>(d->H) * d->d_h, KVD = static_cast<size_t>(d->H_kv) * d->d_h;
  w.w_bytes = f16_weights ? round_up(HD * d->D * 2, 256) + round_up(2 * KVD * d->D * 2, 256) +
                                round_up(HD * d->D * 2, 256)
                          : 0;
  w.sched_bytes = kAttnSchedBytes;
  w.total = w.q_bytes + w.kv_bytes + w.w_bytes + w.sched_bytes;
  return w;
}

// Q' and [K'|V] of M token rows: the Q and KV projections in one GEMM launch
// with QK-norm, RoPE and the query scale fused into its epilogue when the
// head vectors tile the 256-wide output tiles (every Gemma 3 shape with more
// than 16 rows), else the two projections followed by the prologue kernel.
// With `cache` (a CacheRows with Kc set) the prologue kernel also writes the
// rows to their cache slots, and *cache_done tells whether it ran (the fused
// GEMM does not write the cache).
cudaError_t project_qk(const void* x, long ldx, int act_dtype, const void* Wq, const void* Wkv,
                       void* qbuf, void* kvbuf, const void* gamma_q, const void* gamma_k,
                       const int32_t* pos, int M, int D, int H, int H_kv, int d_h,
                       double rope_base, double rope_scale, float query_scale, cudaStream_t s,
                       int* st, const CacheRows* cache = nullptr, bool* cache_done = nullptr,
                       const int32_t* pad_lens = nullptr, int seg_T = 0) {
  if (cache_done != nullptr) *cache_done = false;
  const int HD = H * d_h, KVD = H_kv * d_h;
  if (linear_qknorm_fusable(M, HD, HD, d_h) && linear_qknorm_fusable(M, 2 * KVD, KVD, d_h))
    return launch_qkv_qknorm(x, ldx, Wq, Wkv, D, qbuf, HD, kvbuf, 2 * KVD, M, HD, KVD, D, act_dtype,
                             gamma_q, gamma_k, pos, d_h, rope_base, rope_scale, query_scale, s,
                             st, pad_lens, seg_T);
  cudaError_t e;
  if (M <= kSkinnyMaxRows) {
    // A decode step: both projections in one launch of the few-row kernel.
    e = launch_linear_skinny2(x, ldx, Wq, D, qbuf, HD, HD, Wkv, D, kvbuf, 2 * KVD, 2 * KVD, M, D,
                              act_dtype, kF16, s, st);
  } else {
    // (pad-only tiles: V zeroed for the attention kernels' tile edges)
    e = launch_linear(x, ldx, Wq, D, qbuf, HD, M, HD, D, act_dtype, kF16, s, st, 0, pad_lens,
                      seg_T);
    if (e != cudaSuccess) return e;
    e = launch_linear(x, ldx, Wkv, D, kvbuf, 2 * KVD, M, 2 * KVD, D, act_dtype, kF16, s, st, 0,
                      pad_lens, seg_T, /*zero_pad_tiles=*/true);
  }
  if (e != cudaSuccess) return e;
  e = launch_qk_norm_rope(qbuf, HD, kvbuf, 2 * KVD, gamma_q, gamma_k, pos, M, H, H_kv, d_h,
                          rope_base, rope_scale, query_scale, s,
                          cache != nullptr ? *cache : CacheRows{});
  if (e == cudaSuccess && cache != nullptr && cache_done != nullptr) *cache_done = true;
  return e;
}

// The layer pipeline shared by the single-layer and block entry points.
// act_dtype kBF16: x and the weights are used as given (bf16) and O is bf16.
// act_dtype kF16: x is fp16, the weights are first cast to fp16 copies in the
// workspace, and O is fp16 (about 8x finer rounding of the activations, used
// where layers are stacked and rounding errors accumulate).
int attn_pipeline(const gemma3_attn_dims* d, const void* x, int act_dtype,
                  const int32_t* segment_pos, const int32_t* pad_lens, const void* Wq,
                  const void* Wkv, const void* Wo, const void* gamma_q, const void* gamma_k,
                  int attn_type, int window, double rope_base, double rope_scale,
                  float query_scale, void* out, int out_dtype, uint8_t* ws, cudaStream_t s,
                  bool zero_pad_out) {
  int* st = status_ptr();
  if (st == nullptr) return GEMMA3_ERR_CUDA;
  const int M = d->B * d->T;
  const int HD = d->H * d->d_h, KVD = d->H_kv * d->d_h;
  const bool f16 = act_dtype == kF16;
  const AttnWs w = attn_ws(d, f16);
  void* qbuf = ws;                // Q then Q' (fp16), then O, [M, H*d_h]
  void* kvbuf = ws + w.q_bytes;   // [K'|V] fp16, [M, 2*H_kv*d_h]
  // The attention's work counter is zeroed first, so that the projection,
  // attention and output-projection kernels follow each other directly.
  void* sched = ws + w.q_bytes + w.kv_bytes + w.w_bytes;
  if (cudaMemsetAsync(sched, 0, sizeof(unsigned int), s) != cudaSuccess) return GEMMA3_ERR_CUDA;
  cudaError_t e;
  if (f16) {
    uint8_t* wb = ws + w.q_bytes + w.kv_bytes;
    void* wq = wb;
    void* wkv = wb + round_up(static_cast<size_t>(HD) * d->D * 2, 256);
    void* wo = static_cast<uint8_t*>(wkv) + round_up(static_cast<size_t>(2) * KVD * d->D * 2, 256);
    if (launch_cast_bf16_f16(Wq, wq, static_cast<size_t>(HD) * d->D, s) != cudaSuccess ||
        launch_cast_bf16_f16(Wkv, wkv, static_cast<size_t>(2) * KVD * d->D, s) != cudaSuccess ||
        launch_cast_bf16_f16(Wo, wo, static_cast<size_t>(HD) * d->D, s) != cudaSuccess)
      return GEMMA3_ERR_CUDA;
    Wq = wq;
    Wkv = wkv;
    Wo = wo;
  }
  // Tiles of pad rows only are skipped by both projections (their Q', K', V
  // and output rows are zeros: no valid query or key reads them).
  e = project_qk(x, d->D, act_dtype, Wq, Wkv, qbuf, kvbuf, gamma_q, gamma_k, segment_pos, M,
                 d->D, d->H, d->H_kv, d->d_h, rope_base, rope_scale, query_scale, s, st, nullptr,
                 nullptr, pad_lens, d->T);
  if (e != cudaSuccess) return GEMMA3_ERR_CUDA;
  const int win = attn_type == GEMMA3_LOCAL_SLIDING ? window : 0;
  e = launch_flash_attention(qbuf, kvbuf, static_cast<uint8_t*>(kvbuf) + KVD * 2, 2 * KVD, qbuf,
                             act_dtype, pad_lens, d->B, d->T, d->H, d->H_kv, d->d_h, win, sched, s,
                             st, /*sched_zeroed=*/true);
  if (e != cudaSuccess) return GEMMA3_ERR_CUDA;
  // The layer's output has zero pad rows; a block's attention output is
  // read only on valid rows (its post-norm passes pad rows through).
  e = launch_linear(qbuf, HD, Wo, HD, out, d->D, M, d->D, HD, act_dtype, out_dtype, s, st, 0,
                    pad_lens, d->T, zero_pad_out);
  return to_status(e);
}

int validate_layer_args(const gemma3_attn_dims* dims, const void* x, const int32_t* segment_pos,
                        const void* Wq, const void* Wkv, const void* Wo, const void* gamma_q,
                        const void* gamma_k, int attn_type, int window, double rope_base,
                        double rope_scale, void* workspace) {
  int rc = validate_dims(dims);
  if (rc != GEMMA3_OK) return rc;
  if (!x || !segment_pos || !Wq || !Wkv || !Wo || !gamma_q || !gamma_k || !workspace)
    return GEMMA3_ERR_INVALID_ARG;
  if (attn_type != GEMMA3_LOCAL_SLIDING && attn_type != GEMMA3_GLOBAL)
    return GEMMA3_ERR_INVALID_ARG;
  if (attn_type == GEMMA3_LOCAL_SLIDING && window < 1) return GEMMA3_ERR_INVALID_ARG;
  if (!(rope_base > 0.0) || !(rope_scale > 0.0) || !std::isfinite(rope_base) ||
      !std::isfinite(rope_scale))
    return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wq) || !aligned16(Wkv) || !aligned16(Wo) ||
      !aligned16(gamma_q) || !aligned16(gamma_k) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return GEMMA3_ERR_MISALIGNED;
  return check_device();
}

__global__ void wait_forever_kernel(long long timeout_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nothing arrives on `bar`: the wait must end by its time limit.
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(smem_u32(&bar), 0)) {
      if (globaltimer() - t0 > static_cast<uint64_t>(timeout_ns)) {
        record_error(status, kDevErrTimeoutBase + 99);
        break;
      }
    }
  }
}

}  // namespace

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr) return false;
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) gs[i] = strides_bytes[i];
  }
  const CUresult r = g_encode(map, dt, rank, const_cast<void*>(base), gd, gs, bx, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

namespace {
std::mutex g_prepare_mu;
std::map<std::pair<const void*, int>, int> g_prepared;   // (kernel, device) -> registers
}  // namespace

cudaError_t prepare_kernel(const void* kern, int smem_bytes, int* regs) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_prepare_mu);
  auto it = g_prepared.find({kern, dev});
  if (it == g_prepared.end()) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    it = g_prepared.emplace(std::make_pair(kern, dev), fa.numRegs).first;
  }
  if (regs != nullptr) *regs = it->second;
  return cudaSuccess;
}

}  // namespace g3

using namespace g3;

extern "C" {

int gemma3_layer_attn_type(int layer, int num_layers) {
  if (num_layers < 1 || layer < 0 || layer >= num_layers) return GEMMA3_ERR_INVALID_ARG;
  // Full tiles repeat P; the last N % 6 layers are the prefix P[:N % 6], whose
  // index is again layer % 6 (and never reaches the global slot 5).
  return (layer % 6 == 5) ? GEMMA3_GLOBAL : GEMMA3_LOCAL_SLIDING;
}

int gemma3_layer_config(int layer, int num_layers, int model_size, int* attn_type, int* window,
                        double* rope_base, double* rope_scale) {
  const int t = gemma3_layer_attn_type(layer, num_layers);
  if (t < 0) return t;
  if (model_size < GEMMA3_270M || model_size > GEMMA3_27B) return GEMMA3_ERR_INVALID_ARG;
  const bool small = model_size == GEMMA3_270M || model_size == GEMMA3_1B;
  if (attn_type) *attn_type = t;
  if (t == GEMMA3_LOCAL_SLIDING) {
    if (window) *window = small ? 512 : 1024;
    if (rope_base) *rope_base = 1e4;
    if (rope_scale) *rope_scale = 1.0;
  } else {
    if (window) *window = 0;
    if (rope_base) *rope_base = 1e6;
    if (rope_scale) *rope_scale = small ? 1.0 : 8.0;
  }
  return t;
}

int gemma3_query_scale(int model_size, int D, int H, int d_h, float* alpha) {
  if (alpha == nullptr || D < 1 || H < 1 || d_h < 1) return GEMMA3_ERR_INVALID_ARG;
  if (model_size < GEMMA3_270M || model_size > GEMMA3_27B) return GEMMA3_ERR_INVALID_ARG;
  const double a = model_size == GEMMA3_27B ? 1.0 / std::sqrt(static_cast<double>(D) / H)
                                            : 1.0 / std::sqrt(static_cast<double>(d_h));
  *alpha = static_cast<float>(a);
  return GEMMA3_OK;
}

int gemma3_attn_workspace_size(const gemma3_attn_dims* dims, size_t* bytes) {
  const int rc = validate_dims(dims);
  if (rc != GEMMA3_OK) return rc;
  if (bytes == nullptr) return GEMMA3_ERR_INVALID_ARG;
  *bytes = attn_ws(dims).total;
  return GEMMA3_OK;
}

int gemma3_attn_forward(const gemma3_attn_dims* dims, const void* x, const int32_t* segment_pos,
                        const int32_t* pad_lens, const void* Wq, const void* Wkv, const void* Wo,
                        const void* gamma_q, const void* gamma_k, int attn_type, int window,
                        double rope_base, double rope_scale, float query_scale, void* out,
                        void* workspace, size_t workspace_bytes, void* stream) {
  int rc = validate_layer_args(dims, x, segment_pos, Wq, Wkv, Wo, gamma_q, gamma_k, attn_type,
                               window, rope_base, rope_scale, workspace);
  if (rc != GEMMA3_OK) return rc;
  if (out == nullptr) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(out)) return GEMMA3_ERR_MISALIGNED;
  if (workspace_bytes < attn_ws(dims).total) return GEMMA3_ERR_WORKSPACE;
  return attn_pipeline(dims, x, kBF16, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q, gamma_k,
                       attn_type, window, rope_base, rope_scale, query_scale, out, kBF16,
                       static_cast<uint8_t*>(workspace), as_stream(stream),
                       /*zero_pad_out=*/true);
}

int gemma3_block_attn_workspace_size(const gemma3_attn_dims* dims, size_t* bytes) {
  const int rc = validate_dims(dims);
  if (rc != GEMMA3_OK) return rc;
  if (bytes == nullptr) return GEMMA3_ERR_INVALID_ARG;
  const size_t M = static_cast<size_t>(dims->B) * dims->T;
  *bytes = attn_ws(dims, true).total + round_up(M * dims->D * 2, 256) +
           round_up(M * dims->D * 4, 256);
  return GEMMA3_OK;
}

int gemma3_block_attn_forward(const gemma3_attn_dims* dims, const void* x, int x_dtype,
                              float* y, const int32_t* segment_pos, const int32_t* pad_lens,
                              const void* Wq, const void* Wkv, const void* Wo,
                              const void* gamma_q, const void* gamma_k, const void* gamma_pre,
                              const void* gamma_post, int attn_type, int window,
                              double rope_base, double rope_scale, float query_scale,
                              void* workspace, size_t workspace_bytes, void* stream) {
  int rc = validate_layer_args(dims, x, segment_pos, Wq, Wkv, Wo, gamma_q, gamma_k, attn_type,
                               window, rope_base, rope_scale, workspace);
  if (rc != GEMMA3_OK) return rc;
  if (y == nullptr || gamma_pre == nullptr || gamma_post == nullptr) return GEMMA3_ERR_INVALID_ARG;
  if (x_dtype != GEMMA3_BF16 && x_dtype != GEMMA3_F32) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(gamma_pre) || !aligned16(gamma_post)) return GEMMA3_ERR_MISALIGNED;
  size_t need = 0;
  gemma3_block_attn_workspace_size(dims, &need);
  if (workspace_bytes < need) return GEMMA3_ERR_WORKSPACE;
  const int M = dims->B * dims->T;
  const size_t a_ws = attn_ws(dims, true).total;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* u = ws + a_ws;                                                    // fp16 [M, D]
  float* a = reinterpret_cast<float*>(ws + a_ws + round_up(static_cast<size_t>(M) * dims->D * 2, 256));
  cudaStream_t s = as_stream(stream);
  const int xt = x_dtype == GEMMA3_F32 ? kF32 : kBF16;
  // Pad rows: the pre-norm skips the tiles the projections skip, and the
  // post-norm passes them through (their attention output is zero).
  PadRows pad;
  pad.pad_lens = pad_lens;
  pad.seg_T = dims->T;
  if (launch_rmsnorm_rows(x, xt, gamma_pre, u, kF16, M, dims->D, s, pad) != cudaSuccess)
    return GEMMA3_ERR_CUDA;
  rc = attn_pipeline(dims, u, kF16, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q, gamma_k,
                     attn_type, window, rope_base, rope_scale, query_scale, a, kF32, ws, s,
                     /*zero_pad_out=*/false);
  if (rc != GEMMA3_OK) return rc;
  return to_status(launch_postnorm_residual(a, x, xt, gamma_post, y, M, dims->D, s, pad));
}

// ------------------------------------------------------------ feed-forward half

namespace {

struct FfnWs {
  size_t u, z, m, wgu, wd, total;
};

FfnWs ffn_ws(int M, int D, int D_ff) {
  FfnWs w;
  w.u = round_up(static_cast<size_t>(M) * D * 2, 256);
  w.z = round_up(static_cast<size_t>(M) * D_ff * 2, 256);
  w.m = round_up(static_cast<size_t>(M) * D * 4, 256);
  w.wgu = round_up(static_cast<size_t>(2) * D_ff * D * 2, 256);
  w.wd = round_up(static_cast<size_t>(D) * D_ff * 2, 256);
  w.total = w.u + w.z + w.m + w.wgu + w.wd;
  return w;
}

int validate_ffn(int M, int D, int D_ff) {
  if (M < 1 || D < 8 || D_ff < 8 || D % 8 || D_ff % 8) return GEMMA3_ERR_INVALID_ARG;
  if (static_cast<long long>(M) * D_ff >= (1LL << 40)) return GEMMA3_ERR_INVALID_ARG;
  return GEMMA3_OK;
}

// y = h + RMSNorm_post(FFN(RMSNorm_pre(h))) on fp16 activations (see the
// block path's precision note) with fp32 h / y.
int ffn_pipeline(int M, int D, int D_ff, const void* h, int h_dtype, float* y,
                 const void* gamma_pre, const void* gamma_post, const void* W_gating,
                 const void* W_down, uint8_t* ws, cudaStream_t s) {
  int* st = status_ptr();
  if (st == nullptr) return GEMMA3_ERR_CUDA;
  const FfnWs w = ffn_ws(M, D, D_ff);
  uint8_t* u = ws;
  uint8_t* z = u + w.u;
  float* m = reinterpret_cast<float*>(z + w.z);
  uint8_t* wgu = z + w.z + w.m;
  uint8_t* wd = wgu + w.wgu;
  if (launch_rmsnorm_rows(h, h_dtype, gamma_pre, u, kF16, M, D, s) != cudaSuccess ||
      launch_cast_bf16_f16(W_gating, wgu, static_cast<size_t>(2) * D_ff * D, s) != cudaSuccess ||
      launch_cast_bf16_f16(W_down, wd, static_cast<size_t>(D) * D_ff, s) != cudaSuccess ||
      launch_geglu(u, D, wgu, D, z, D_ff, M, D_ff, D, kF16, s, st) != cudaSuccess ||
      launch_linear(z, D_ff, wd, D_ff, m, D, M, D, D_ff, kF16, kF32, s, st, 0) != cudaSuccess)
    return GEMMA3_ERR_CUDA;
  return to_status(launch_postnorm_residual(m, h, h_dtype, gamma_post, y, M, D, s));
}

}  // namespace

int gemma3_block_ffn_workspace_size(int M, int D, int D_ff, size_t* bytes) {
  const int rc = validate_ffn(M, D, D_ff);
  if (rc != GEMMA3_OK) return rc;
  if (bytes == nullptr) return GEMMA3_ERR_INVALID_ARG;
  *bytes = ffn_ws(M, D, D_ff).total;
  return GEMMA3_OK;
}

int gemma3_block_ffn_forward(int M, int D, int D_ff, const float* h, float* y,
                             const void* gamma_pre_ffn, const void* gamma_post_ffn,
                             const void* W_gating, const void* W_down, void* workspace,
                             size_t workspace_bytes, void* stream) {
  int rc = validate_ffn(M, D, D_ff);
  if (rc != GEMMA3_OK) return rc;
  if (!h || !y || !gamma_pre_ffn || !gamma_post_ffn || !W_gating || !W_down || !workspace)
    return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(y) || !aligned16(gamma_pre_ffn) || !aligned16(gamma_post_ffn) ||
      !aligned16(W_gating) || !aligned16(W_down) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return GEMMA3_ERR_MISALIGNED;
  if (workspace_bytes < ffn_ws(M, D, D_ff).total) return GEMMA3_ERR_WORKSPACE;
  rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  return ffn_pipeline(M, D, D_ff, h, kF32, y, gamma_pre_ffn, gamma_post_ffn, W_gating, W_down,
                      static_cast<uint8_t*>(workspace), as_stream(stream));
}

int gemma3_block_workspace_size(const gemma3_attn_dims* dims, int D_ff, size_t* bytes) {
  if (bytes == nullptr) return GEMMA3_ERR_INVALID_ARG;
  size_t a = 0, f = 0;
  int rc = gemma3_block_attn_workspace_size(dims, &a);
  if (rc != GEMMA3_OK) return rc;
  rc = gemma3_block_ffn_workspace_size(dims->B * dims->T, dims->D, D_ff, &f);
  if (rc != GEMMA3_OK) return rc;
  *bytes = a > f ? a : f;
  return GEMMA3_OK;
}

int gemma3_block_forward(const gemma3_attn_dims* dims, int D_ff, const void* x, int x_dtype,
                         float* y, const int32_t* segment_pos, const int32_t* pad_lens,
                         const void* Wq, const void* Wkv, const void* Wo, const void* gamma_q,
                         const void* gamma_k, const void* gamma_pre_attn,
                         const void* gamma_post_attn, const void* gamma_pre_ffn,
                         const void* gamma_post_ffn, const void* W_gating, const void* W_down,
                         int attn_type, int window, double rope_base, double rope_scale,
                         float query_scale, void* workspace, size_t workspace_bytes,
                         void* stream) {
  size_t need = 0;
  int rc = gemma3_block_workspace_size(dims, D_ff, &need);
  if (rc != GEMMA3_OK) return rc;
  if (!gamma_pre_ffn || !gamma_post_ffn || !W_gating || !W_down) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(gamma_pre_ffn) || !aligned16(gamma_post_ffn) || !aligned16(W_gating) ||
      !aligned16(W_down))
    return GEMMA3_ERR_MISALIGNED;
  if (workspace_bytes < need) return GEMMA3_ERR_WORKSPACE;
  // h = x + RMSNorm_post-attn(Attn(RMSNorm_pre-attn(x))) into y, then the
  // feed-forward sandwich in place on y (the workspace is reused in turn).
  rc = gemma3_block_attn_forward(dims, x, x_dtype, y, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q,
                                 gamma_k, gamma_pre_attn, gamma_post_attn, attn_type, window,
                                 rope_base, rope_scale, query_scale, workspace, workspace_bytes,
                                 stream);
  if (rc != GEMMA3_OK) return rc;
  return ffn_pipeline(dims->B * dims->T, dims->D, D_ff, y, kF32, y, gamma_pre_ffn,
                      gamma_post_ffn, W_gating, W_down, static_cast<uint8_t*>(workspace),
                      as_stream(stream));
}

// ------------------------------------------------------------ the model

namespace {

struct ModelWs {
  size_t x, h, block, total;
};

int model_ws(const gemma3_attn_dims* d, int D_ff, ModelWs* w) {
  size_t blk = 0;
  const int rc = gemma3_block_workspace_size(d, D_ff, &blk);
  if (rc != GEMMA3_OK) return rc;
  const size_t M = static_cast<size_t>(d->B) * d->T;
  w->x = round_up(M * d->D * 4, 256);
  w->h = round_up(M * d->D * 2, 256);
  w->block = round_up(blk, 256);
  w->total = w->x + w->h + w->block;
  return GEMMA3_OK;
}

}  // namespace

int gemma3_model_workspace_size(const gemma3_attn_dims* dims, int D_ff, int V, size_t* bytes) {
  if (bytes == nullptr || V < 1) return GEMMA3_ERR_INVALID_ARG;
  ModelWs w;
  const int rc = model_ws(dims, D_ff, &w);
  if (rc != GEMMA3_OK) return rc;
  *bytes = w.total;
  return GEMMA3_OK;
}

int gemma3_embed(const int32_t* tokens, const void* E, int V, int D, int M, float scale, float* x,
                 void* stream) {
  if (!tokens || !E || !x || V < 1 || D < 8 || D % 8 || M < 0) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(E) || !aligned16(x)) return GEMMA3_ERR_MISALIGNED;
  int rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  int* st = status_ptr();
  if (st == nullptr) return GEMMA3_ERR_CUDA;
  return to_status(launch_embed_rows(tokens, E, V, D, M, scale, x, as_stream(stream), st));
}

int gemma3_model_forward(const gemma3_attn_dims* dims, int D_ff, int V, int num_layers,
                         int model_size, const int32_t* tokens, const int32_t* segment_pos,
                         const int32_t* pad_lens, const void* E,
                         const gemma3_block_weights* layers, const void* gamma_final,
                         float* logits, void* workspace, size_t workspace_bytes, void* stream) {
  ModelWs w;
  int rc = validate_dims(dims);
  if (rc != GEMMA3_OK) return rc;
  rc = model_ws(dims, D_ff, &w);
  if (rc != GEMMA3_OK) return rc;
  if (V < 1 || num_layers < 0 || !tokens || !segment_pos || !E || !gamma_final || !logits ||
      !workspace || (num_layers > 0 && !layers))
    return GEMMA3_ERR_INVALID_ARG;
  if (model_size < GEMMA3_270M || model_size > GEMMA3_27B) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(E) || !aligned16(gamma_final) || !aligned16(logits) || V % 4 ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return GEMMA3_ERR_MISALIGNED;
  if (workspace_bytes < w.total) return GEMMA3_ERR_WORKSPACE;
  rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  int* st = status_ptr();
  if (st == nullptr) return GEMMA3_ERR_CUDA;
  float alpha = 0.f;
  rc = gemma3_query_scale(model_size, dims->D, dims->H, dims->d_h, &alpha);
  if (rc != GEMMA3_OK) return rc;
  const int M = dims->B * dims->T, D = dims->D;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* x = reinterpret_cast<float*>(ws);           // residual stream, fp32 [M, D]
  void* h = ws + w.x;                                 // final norm, bf16 [M, D]
  void* bws = ws + w.x + w.h;                         // the blocks' workspace
  cudaStream_t s = as_stream(stream);
  if (launch_embed_rows(tokens, E, V, D, M, static_cast<float>(std::sqrt(static_cast<double>(D))),
                        x, s, st) != cudaSuccess)
    return GEMMA3_ERR_CUDA;
  for (int l = 0; l < num_layers; ++l) {
    int type = 0, window = 0;
    double base = 0.0, scale = 0.0;
    rc = gemma3_layer_config(l, num_layers, model_size, &type, &window, &base, &scale);
    if (rc < 0) return rc;
    const gemma3_block_weights& L = layers[l];
    rc = gemma3_block_forward(dims, D_ff, x, GEMMA3_F32, x, segment_pos, pad_lens, L.Wq, L.Wkv,
                              L.Wo, L.gamma_q, L.gamma_k, L.gamma_pre_attn, L.gamma_post_attn,
                              L.gamma_pre_ffn, L.gamma_post_ffn, L.W_gating, L.W_down, type,
                              window, base, scale, alpha, bws, w.block, stream);
    if (rc != GEMMA3_OK) return rc;
  }
  if (launch_rmsnorm_rows(x, kF32, gamma_final, h, kBF16, M, D, s) != cudaSuccess)
    return GEMMA3_ERR_CUDA;
  return to_status(launch_linear(h, D, E, D, logits, V, M, V, D, kBF16, kF32, s, st, 0));
}

// ------------------------------------------------------------ KV-cache path

namespace {

struct CachedWs {
  size_t q, kv, attn, total;
};

CachedWs cached_ws(const gemma3_attn_dims* d, int S) {
  const size_t M = static_cast<size_t>(d->B) * d->T;
  CachedWs w;
  w.q = round_up(M * d->H * d->d_h * 2, 256);
  w.kv = round_up(M * 2 * d->H_kv * d->d_h * 2, 256);
  w.attn = round_up(cached_attention_ws_bytes(d->B, d->T, S, d->H, d->H_kv, d->d_h), 256) +
           kAttnSchedBytes;
  w.total = w.q + w.kv + w.attn;
  return w;
}

int validate_cache(int B, int T, int S, int end_index, int H_kv, int d_h, const void* K_cache,
                   const void* V_cache, const int32_t* pos_cache) {
  if (!K_cache || !V_cache || !pos_cache) return GEMMA3_ERR_INVALID_ARG;
  if (S < 1 || S > (1 << 30) || end_index < 0 || T < 1 ||
      static_cast<long long>(end_index) + T > S)
    return GEMMA3_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * S >= (1LL << 40) / (static_cast<long long>(H_kv) * d_h))
    return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(K_cache) || !aligned16(V_cache) || (reinterpret_cast<uintptr_t>(pos_cache) & 3u))
    return GEMMA3_ERR_MISALIGNED;
  return GEMMA3_OK;
}

// A prompt written at slot 0 of a global layer sees exactly the causal,
// unpadded part of itself (every later slot is beyond its causal limit), which
// is the mask of the tensor-core flash kernel; from this length on that kernel
// is used for it.
constexpr int kFlashPrefillMinT = 128;

}  // namespace

int gemma3_attn_cached_workspace_size(const gemma3_attn_dims* dims, int S, size_t* bytes) {
  const int rc = validate_dims(dims);
  if (rc != GEMMA3_OK) return rc;
  if (bytes == nullptr || S < 1) return GEMMA3_ERR_INVALID_ARG;
  *bytes = cached_ws(dims, S).total;
  return GEMMA3_OK;
}

int gemma3_attn_forward_cached(const gemma3_attn_dims* dims, int S, int end_index, const void* x,
                               const int32_t* segment_pos, const int32_t* pad_lens,
                               const void* Wq, const void* Wkv, const void* Wo,
                               const void* gamma_q, const void* gamma_k, int attn_type,
                               int window, double rope_base, double rope_scale, float query_scale,
                               void* K_cache, void* V_cache, int32_t* pos_cache, void* out,
                               void* workspace, size_t workspace_bytes, void* stream) {
  int rc = validate_layer_args(dims, x, segment_pos, Wq, Wkv, Wo, gamma_q, gamma_k, attn_type,
                               window, rope_base, rope_scale, workspace);
  if (rc != GEMMA3_OK) return rc;
  rc = validate_cache(dims->B, dims->T, S, end_index, dims->H_kv, dims->d_h, K_cache, V_cache,
                      pos_cache);
  if (rc != GEMMA3_OK) return rc;
  if (out == nullptr) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(out)) return GEMMA3_ERR_MISALIGNED;
  const CachedWs w = cached_ws(dims, S);
  if (workspace_bytes < w.total) return GEMMA3_ERR_WORKSPACE;
  int* st = status_ptr();
  if (st == nullptr) return GEMMA3_ERR_CUDA;
  const gemma3_attn_dims* d = dims;
  const int M = d->B * d->T;
  const int HD = d->H * d->d_h, KVD = d->H_kv * d->d_h;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* qbuf = ws;                 // Q, then Q', then O  [M, H*d_h] fp16/bf16
  uint8_t* kvbuf = ws + w.q;          // [K'|V] fp16  [M, 2*KVD]
  uint8_t* aws = kvbuf + w.kv;        // attention partials
  cudaStream_t s = as_stream(stream);
  // The new K'/V rows go to the cache from the prologue kernel when it runs
  // on its own (a decode step), else by the append kernel.
  CacheRows cr;
  cr.Kc = K_cache;
  cr.Vc = V_cache;
  cr.posc = pos_cache;
  cr.V = kvbuf + KVD * 2;
  cr.ldv = 2 * KVD;
  cr.pad_lens = pad_lens;
  cr.T = d->T;
  cr.S = S;
  cr.end = end_index;
  const bool flash = end_index == 0 && attn_type == GEMMA3_GLOBAL && d->T >= kFlashPrefillMinT;
  if (!flash && attn_type == GEMMA3_LOCAL_SLIDING) {
    // A prologue kernel that writes the cache also scans the local layer's
    // cache span for the cache attention, in the same launch.
    cr.span_part = cached_attention_layout(aws, d->B, d->T, S, d->H, d->H_kv, d->d_h).span_part;
    cr.window = window;
    cr.nchunk = cached_span_chunks(d->T, end_index);
  }
  bool cached = false;
  if (project_qk(x, d->D, kBF16, Wq, Wkv, qbuf, kvbuf, gamma_q, gamma_k, segment_pos, M, d->D,
                 d->H, d->H_kv, d->d_h, rope_base, rope_scale, query_scale, s, st, &cr,
                 &cached) != cudaSuccess ||
      (!cached &&
       launch_kv_cache_append(kvbuf, kvbuf + KVD * 2, 2 * KVD, segment_pos, pad_lens, d->B, d->T, S,
                              end_index, KVD, K_cache, V_cache, pos_cache, s) != cudaSuccess))
    return GEMMA3_ERR_CUDA;
  cudaError_t e;
  if (flash)
    e = launch_flash_attention(qbuf, kvbuf, kvbuf + KVD * 2, 2 * KVD, qbuf, kBF16, pad_lens, d->B,
                               d->T, d->H, d->H_kv, d->d_h, 0, aws + w.attn - kAttnSchedBytes, s,
                               st);
  else
    e = launch_cached_attention(qbuf, K_cache, V_cache, pos_cache, segment_pos, pad_lens, qbuf,
                                kBF16, d->B, d->T, S, end_index, d->H, d->H_kv, d->d_h,
                                attn_type == GEMMA3_LOCAL_SLIDING ? window : 0, aws, s, st,
                                /*prepared=*/cached);
  if (e != cudaSuccess) return GEMMA3_ERR_CUDA;
  return to_status(launch_linear(qbuf, HD, Wo, HD, out, d->D, M, d->D, HD, kBF16, kBF16, s, st, 0));
}

int gemma3_kv_cache_write(const void* K_rows, const void* V_rows, long ld_rows,
                          const int32_t* segment_pos, const int32_t* pad_lens, int B, int T,
                          int S, int end_index, int H_kv, int d_h, void* K_cache, void* V_cache,
                          int32_t* pos_cache, void* stream) {
  if (!K_rows || !V_rows || !segment_pos || B < 1 || H_kv < 1) return GEMMA3_ERR_INVALID_ARG;
  if (d_h != 128 && d_h != 256) return GEMMA3_ERR_UNSUPPORTED;
  int rc = validate_cache(B, T, S, end_index, H_kv, d_h, K_cache, V_cache, pos_cache);
  if (rc != GEMMA3_OK) return rc;
  if (ld_rows < static_cast<long>(H_kv) * d_h) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(K_rows) || !aligned16(V_rows) || (ld_rows * 2) % 16) return GEMMA3_ERR_MISALIGNED;
  rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  return to_status(launch_kv_cache_append(K_rows, V_rows, ld_rows, segment_pos, pad_lens, B, T, S,
                                          end_index, H_kv * d_h, K_cache, V_cache, pos_cache,
                                          as_stream(stream)));
}

int gemma3_cached_attention_workspace_size(int B, int T, int S, int H, int H_kv, int d_h,
                                           size_t* bytes) {
  if (bytes == nullptr || B < 1 || T < 1 || S < 1 || H < 1 || H_kv < 1 || H % H_kv)
    return GEMMA3_ERR_INVALID_ARG;
  const int G = H / H_kv;
  if ((d_h != 128 && d_h != 256) || (G != 1 && G != 2 && G != 4)) return GEMMA3_ERR_UNSUPPORTED;
  *bytes = round_up(cached_attention_ws_bytes(B, T, S, H, H_kv, d_h), 256);
  return GEMMA3_OK;
}

int gemma3_cached_attention(const void* Q, const void* K_cache, const void* V_cache,
                            const int32_t* pos_cache, const int32_t* segment_pos,
                            const int32_t* pad_lens, void* O, int o_dtype, int B, int T, int S,
                            int end_index, int H, int H_kv, int d_h, int window, void* workspace,
                            size_t workspace_bytes, void* stream) {
  size_t need = 0;
  int rc = gemma3_cached_attention_workspace_size(B, T, S, H, H_kv, d_h, &need);
  if (rc != GEMMA3_OK) return rc;
  if (!Q || !O || !segment_pos || !workspace) return GEMMA3_ERR_INVALID_ARG;
  if (o_dtype != GEMMA3_BF16 && o_dtype != GEMMA3_F16) return GEMMA3_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * T * H >= (1LL << 31)) return GEMMA3_ERR_INVALID_ARG;
  rc = validate_cache(B, T, S, end_index, H_kv, d_h, K_cache, V_cache, pos_cache);
  if (rc != GEMMA3_OK) return rc;
  if (!aligned16(Q) || !aligned16(O) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return GEMMA3_ERR_MISALIGNED;
  if (workspace_bytes < need) return GEMMA3_ERR_WORKSPACE;
  rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  int* st = status_ptr();
  if (st == nullptr) return GEMMA3_ERR_CUDA;
  return to_status(launch_cached_attention(Q, K_cache, V_cache, pos_cache, segment_pos, pad_lens, O,
                                           o_dtype == GEMMA3_F16 ? kF16 : kBF16, B, T, S,
                                           end_index, H, H_kv, d_h, window > 0 ? window : 0,
                                           workspace, as_stream(stream), st));
}

int gemma3_geglu(const void* A, long lda, const void* W_gating, long ldw, void* Z, long ldz,
                 int M, int D_ff, int K, int in_dtype, void* stream) {
  if (!A || !W_gating || !Z || M < 0 || D_ff < 1 || K < 1) return GEMMA3_ERR_INVALID_ARG;
  if (in_dtype != GEMMA3_BF16 && in_dtype != GEMMA3_F16) return GEMMA3_ERR_INVALID_ARG;
  if (lda < K || ldw < K || ldz < D_ff) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W_gating) || !aligned16(Z) || (lda * 2) % 16 ||
      (ldw * 2) % 16 || (ldz * 2) % 16)
    return GEMMA3_ERR_MISALIGNED;
  int rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  int* st = status_ptr();
  if (st == nullptr) return GEMMA3_ERR_CUDA;
  return to_status(launch_geglu(A, lda, W_gating, ldw, Z, ldz, M, D_ff, K,
                                in_dtype == GEMMA3_F16 ? kF16 : kBF16, as_stream(stream), st));
}

int gemma3_set_gemm_tile_rows(int rows) {
  const int prev = set_gemm_tile_rows(rows);
  return prev < 0 ? GEMMA3_ERR_INVALID_ARG : prev;
}

int gemma3_linear(const void* A, long lda, const void* W, long ldw, void* C, long ldc, int M,
                  int N, int K, int in_dtype, int out_dtype, int max_ctas,
                  const int32_t* pad_lens, int seg_T, void* stream) {
  if (!A || !W || !C || M < 0 || N < 0 || K < 1) return GEMMA3_ERR_INVALID_ARG;
  if (pad_lens != nullptr && (seg_T < 1 || M % seg_T != 0)) return GEMMA3_ERR_INVALID_ARG;
  if (in_dtype != GEMMA3_BF16 && in_dtype != GEMMA3_F16) return GEMMA3_ERR_INVALID_ARG;
  if (out_dtype != GEMMA3_BF16 && out_dtype != GEMMA3_F16 && out_dtype != GEMMA3_F32)
    return GEMMA3_ERR_INVALID_ARG;
  if (lda < K || ldw < K || ldc < N) return GEMMA3_ERR_INVALID_ARG;
  const int osz = out_dtype == GEMMA3_F32 ? 4 : 2;
  if (!aligned16(A) || !aligned16(W) || !aligned16(C) || (lda * 2) % 16 || (ldw * 2) % 16 ||
      (ldc * osz) % 16)
    return GEMMA3_ERR_MISALIGNED;
  int rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  int* st = status_ptr();
  if (st == nullptr) return GEMMA3_ERR_CUDA;
  const int it = in_dtype == GEMMA3_F16 ? kF16 : kBF16;
  const int dt = out_dtype == GEMMA3_F32 ? kF32 : (out_dtype == GEMMA3_F16 ? kF16 : kBF16);
  return to_status(launch_linear(A, lda, W, ldw, C, ldc, M, N, K, it, dt, as_stream(stream), st,
                                 max_ctas, pad_lens, pad_lens != nullptr ? seg_T : 0));
}

int gemma3_qkv_proj_norm_rope(const void* x, long ldx, const void* Wq, const void* Wkv, void* Q,
                              void* KV, int M, int D, int H, int H_kv, int d_h, int in_dtype,
                              const void* gamma_q, const void* gamma_k, const int32_t* pos,
                              double rope_base, double rope_scale, float query_scale,
                              const int32_t* pad_lens, int seg_T, void* stream) {
  if (!x || !Wq || !Wkv || !Q || !KV || !gamma_q || !gamma_k || !pos || M < 0 || D < 8 ||
      D % 8 || H < 1 || H_kv < 1)
    return GEMMA3_ERR_INVALID_ARG;
  if (pad_lens != nullptr && (seg_T < 1 || M % seg_T != 0)) return GEMMA3_ERR_INVALID_ARG;
  if (d_h != 128 && d_h != 256) return GEMMA3_ERR_UNSUPPORTED;
  if (in_dtype != GEMMA3_BF16 && in_dtype != GEMMA3_F16) return GEMMA3_ERR_INVALID_ARG;
  if (ldx < D) return GEMMA3_ERR_INVALID_ARG;
  if (!(rope_base > 0.0) || !(rope_scale > 0.0)) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wq) || !aligned16(Wkv) || !aligned16(Q) || !aligned16(KV) ||
      !aligned16(gamma_q) || !aligned16(gamma_k) || (ldx * 2) % 16)
    return GEMMA3_ERR_MISALIGNED;
  int rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  int* st = status_ptr();
  if (st == nullptr) return GEMMA3_ERR_CUDA;
  return to_status(project_qk(x, ldx, in_dtype == GEMMA3_F16 ? kF16 : kBF16, Wq, Wkv, Q, KV,
                              gamma_q, gamma_k, pos, M, D, H, H_kv, d_h, rope_base, rope_scale,
                              query_scale, as_stream(stream), st, nullptr, nullptr, pad_lens,
                              pad_lens != nullptr ? seg_T : 0));
}

int gemma3_linear_qk_norm_rope(const void* A, long lda, const void* W, long ldw, void* C,
                               long ldc, int M, int N, int K, int in_dtype, const void* gamma,
                               const int32_t* pos, int d_h, int n_norm, double rope_base,
                               double rope_scale, float scale, void* stream) {
  if (!A || !W || !C || !gamma || !pos || M < 0 || N < 1 || K < 1) return GEMMA3_ERR_INVALID_ARG;
  if (in_dtype != GEMMA3_BF16 && in_dtype != GEMMA3_F16) return GEMMA3_ERR_INVALID_ARG;
  if (lda < K || ldw < K || ldc < N) return GEMMA3_ERR_INVALID_ARG;
  if (!(rope_base > 0.0) || !(rope_scale > 0.0)) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(C) || !aligned16(gamma) || (lda * 2) % 16 ||
      (ldw * 2) % 16 || (ldc * 2) % 16)
    return GEMMA3_ERR_MISALIGNED;
  if (M > 0 && !linear_qknorm_fusable(M, N, n_norm, d_h)) return GEMMA3_ERR_UNSUPPORTED;
  int rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  int* st = status_ptr();
  if (st == nullptr) return GEMMA3_ERR_CUDA;
  return to_status(launch_linear_qknorm(A, lda, W, ldw, C, ldc, M, N, K,
                                        in_dtype == GEMMA3_F16 ? kF16 : kBF16, gamma, pos, d_h,
                                        n_norm, rope_base, rope_scale, scale, as_stream(stream),
                                        st));
}

int gemma3_cast_bf16_f16(const void* src, void* dst, size_t n, void* stream) {
  if (!src || !dst) return GEMMA3_ERR_INVALID_ARG;
  if (n % 8 != 0) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return GEMMA3_ERR_MISALIGNED;
  int rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  return to_status(launch_cast_bf16_f16(src, dst, n, as_stream(stream)));
}

int gemma3_qk_norm_rope(void* Q, long ldq, void* K, long ldk, const void* gamma_q,
                        const void* gamma_k, const int32_t* pos, int M, int H, int H_kv,
                        int d_h, double rope_base, double rope_scale, float query_scale,
                        void* stream) {
  if (!Q || !K || !gamma_q || !gamma_k || !pos || M < 0 || H < 1 || H_kv < 1)
    return GEMMA3_ERR_INVALID_ARG;
  if (d_h != 128 && d_h != 256) return GEMMA3_ERR_UNSUPPORTED;
  if (ldq < static_cast<long>(H) * d_h || ldk < static_cast<long>(H_kv) * d_h)
    return GEMMA3_ERR_INVALID_ARG;
  if (!(rope_base > 0.0) || !(rope_scale > 0.0)) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || (ldq * 2) % 16 || (ldk * 2) % 16 || !aligned16(gamma_q) ||
      !aligned16(gamma_k))
    return GEMMA3_ERR_MISALIGNED;
  int rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  return to_status(launch_qk_norm_rope(Q, ldq, K, ldk, gamma_q, gamma_k, pos, M, H, H_kv, d_h,
                                       rope_base, rope_scale, query_scale, as_stream(stream)));
}

int gemma3_flash_attention(const void* Q, const void* K, const void* V, long ldkv, void* O,
                           int o_dtype, const int32_t* pad_lens, int B, int T, int H, int H_kv,
                           int d_h, int window, void* scratch, void* stream) {
  if (!Q || !K || !V || !O || B < 1 || T < 1 || H < 1 || H_kv < 1 || H % H_kv)
    return GEMMA3_ERR_INVALID_ARG;
  if (o_dtype != GEMMA3_BF16 && o_dtype != GEMMA3_F16) return GEMMA3_ERR_INVALID_ARG;
  const int G = H / H_kv;
  if ((d_h != 128 && d_h != 256) || (G != 1 && G != 2 && G != 4)) return GEMMA3_ERR_UNSUPPORTED;
  if (ldkv < static_cast<long>(H_kv) * d_h) return GEMMA3_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * T >= (1LL << 31)) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || (ldkv * 2) % 16 ||
      !aligned16(scratch))
    return GEMMA3_ERR_MISALIGNED;
  int rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  int* st = status_ptr();
  if (st == nullptr) return GEMMA3_ERR_CUDA;
  return to_status(launch_flash_attention(Q, K, V, ldkv, O, o_dtype == GEMMA3_F16 ? kF16 : kBF16,
                                          pad_lens, B, T, H, H_kv, d_h, window > 0 ? window : 0,
                                          scratch, as_stream(stream), st));
}

int gemma3_rmsnorm(const void* x, int x_dtype, const void* gamma, void* u, int u_dtype, int M,
                   int D, const int32_t* pad_lens, int seg_T, void* stream) {
  if (!x || !gamma || !u || M < 0 || D < 4 || D % 4) return GEMMA3_ERR_INVALID_ARG;
  if (pad_lens != nullptr && (seg_T < 1 || M % seg_T != 0)) return GEMMA3_ERR_INVALID_ARG;
  if (x_dtype != GEMMA3_BF16 && x_dtype != GEMMA3_F32) return GEMMA3_ERR_INVALID_ARG;
  if (u_dtype != GEMMA3_BF16 && u_dtype != GEMMA3_F16) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(gamma) || !aligned16(u)) return GEMMA3_ERR_MISALIGNED;
  int rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  PadRows pad;
  pad.pad_lens = pad_lens;
  pad.seg_T = seg_T;
  return to_status(launch_rmsnorm_rows(x, x_dtype == GEMMA3_F32 ? kF32 : kBF16, gamma, u,
                                       u_dtype == GEMMA3_F16 ? kF16 : kBF16, M, D,
                                       as_stream(stream), pad));
}

int gemma3_postnorm_residual(const float* a, const void* x, int x_dtype, const void* gamma,
                             float* y, int M, int D, const int32_t* pad_lens, int seg_T,
                             void* stream) {
  if (!a || !x || !gamma || !y || M < 0 || D < 4 || D % 4) return GEMMA3_ERR_INVALID_ARG;
  if (pad_lens != nullptr && (seg_T < 1 || M % seg_T != 0)) return GEMMA3_ERR_INVALID_ARG;
  if (x_dtype != GEMMA3_BF16 && x_dtype != GEMMA3_F32) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(x) || !aligned16(gamma) || !aligned16(y))
    return GEMMA3_ERR_MISALIGNED;
  int rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  PadRows pad;
  pad.pad_lens = pad_lens;
  pad.seg_T = seg_T;
  return to_status(launch_postnorm_residual(a, x, x_dtype == GEMMA3_F32 ? kF32 : kBF16, gamma, y,
                                            M, D, as_stream(stream), pad));
}

int gemma3_attn_check_status(void* stream) {
  cudaStream_t s = as_stream(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return GEMMA3_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g3_device_status, sizeof(int)) != cudaSuccess)
    return GEMMA3_ERR_CUDA;
  t_last_device_status = v;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g3_device_status, &zero, sizeof(int)) != cudaSuccess)
      return GEMMA3_ERR_CUDA;
    return v >= kDevErrBadToken ? GEMMA3_ERR_BAD_INPUT : GEMMA3_ERR_TIMEOUT;
  }
  return GEMMA3_OK;
}

int gemma3_last_device_status(void) { return t_last_device_status; }

const char* gemma3_strerror(int status) {
  switch (status) {
    case GEMMA3_OK: return "ok";
    case GEMMA3_ERR_INVALID_ARG: return "invalid argument";
    case GEMMA3_ERR_MISALIGNED: return "pointer or stride not 16-byte aligned";
    case GEMMA3_ERR_UNSUPPORTED: return "unsupported shape or device";
    case GEMMA3_ERR_CUDA: return "CUDA error";
    case GEMMA3_ERR_TIMEOUT: return "kernel gave up on a bounded wait";
    case GEMMA3_ERR_WORKSPACE: return "workspace too small";
    case GEMMA3_ERR_BAD_INPUT: return "a kernel found invalid input data";
    default: return "unknown status";
  }
}

int gemma3_selftest_wait_timeout(long long timeout_ns, void* stream) {
  if (timeout_ns < 1000000LL || timeout_ns > 5000000000LL) return GEMMA3_ERR_INVALID_ARG;
  int rc = check_device();
  if (rc != GEMMA3_OK) return rc;
  int* st = status_ptr();
  if (st == nullptr) return GEMMA3_ERR_CUDA;
  cudaStream_t s = as_stream(stream);
  wait_forever_kernel<<<1, 32, 0, s>>>(timeout_ns, st);
  if (cudaGetLastError() != cudaSuccess) return GEMMA3_ERR_CUDA;
  return gemma3_attn_check_status(stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Forward pass without any device allocation.
//
// Some callers cannot hand the library a workspace: code that runs where
// cudaMalloc is not allowed or not wanted (inside a real-time loop that must
// never hit the allocator, in a host process whose memory is owned by another
// framework's pool, or behind an interface that only passes input and output
// buffers).  For them the layer's intermediate Q/K/V/O rows live in one
// fixed array of device memory that belongs to the library itself.
//
// The array is a file-scope __device__ variable: the CUDA runtime reserves it
// on every GPU that loads this library, for as long as the process runs.  Its
// name is only a host-side stand-in in host code, so the device address is
// looked up once per device with cudaGetSymbolAddress and passed to the
// kernels.  Every call shares this one array: two calls whose kernels overlap
// on the GPU (different streams, or different host threads without ordering)
// race on it and produce garbage.  The kernels overwrite every scratch byte
// they read, so nothing has to be cleared between calls.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
static __device__ __align__(256) unsigned char g3_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (first call on a
// device looks it up; later calls read the cache).  nullptr on failure.
void* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g3_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" size_t gemma3_attn_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

extern "C" int gemma3_attn_forward_noalloc(const gemma3_attn_dims* dims, const void* x,
                                           const int32_t* segment_pos, const int32_t* pad_lens,
                                           const void* Wq, const void* Wkv, const void* Wo,
                                           const void* gamma_q, const void* gamma_k,
                                           int attn_type, int window, double rope_base,
                                           double rope_scale, float query_scale, void* out,
                                           void* stream) {
  const int rc = validate_dims(dims);
  if (rc != GEMMA3_OK) return rc;
  if (out == nullptr) return GEMMA3_ERR_INVALID_ARG;
  if (!aligned16(out)) return GEMMA3_ERR_MISALIGNED;
  if (attn_ws(dims).total > kNoAllocScratchBytes) return GEMMA3_ERR_WORKSPACE;
  // Same validation as the workspace entry point (a non-null stand-in for the
  // workspace pointer: the scratch address is checked separately below).
  const int vr = validate_layer_args(dims, x, segment_pos, Wq, Wkv, Wo, gamma_q, gamma_k,
                                     attn_type, window, rope_base, rope_scale,
                                     reinterpret_cast<void*>(uintptr_t(256)));
  if (vr != GEMMA3_OK) return vr;
  void* scratch = noalloc_scratch();
  if (scratch == nullptr) return GEMMA3_ERR_CUDA;
  return attn_pipeline(dims, x, kBF16, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q, gamma_k,
                       attn_type, window, rope_base, rope_scale, query_scale, out, kBF16,
                       static_cast<uint8_t*>(scratch), as_stream(stream),
                       /*zero_pad_out=*/true);
}
