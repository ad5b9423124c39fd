// C[M, N] = A[M, K] * W[N, K]^T for few rows (M <= 16): the projections of a
// decode step ("Gemma 3 Attention Block", How it works: Projections, with one
// new token per batch row).
//
// With M this small the product does 2*M flops per 2-byte weight, so it is
// bound by reading W once from HBM, and a 128-row tensor-core tile would be
// almost all padding.  The kernel runs on the CUDA cores: each warp owns two
// output columns (two rows of W), its lanes stride K in 16-byte chunks with
// eight chunks of both rows in flight, A (a few KB) is read through L1, the
// sums are fp32, and a warp reduction finishes each output.
#include "internal.h"
#include "ptx.cuh"

namespace g3 {

namespace {

constexpr int kWarps = 4;     // warps per CTA
constexpr int kRows = 2;      // rows of W per warp
constexpr int kUnroll = 8;    // 256-element K chunks in flight per row

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <typename T>
__device__ __forceinline__ void to_f8(const uint4& v, float (&f)[8]);
template <>
__device__ __forceinline__ void to_f8<__nv_bfloat16>(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = __bfloat1622float2(h[i]);
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}
template <>
__device__ __forceinline__ void to_f8<__half>(const uint4& v, float (&f)[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = __half22float2(h[i]);
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}

template <typename OutT>
__device__ __forceinline__ OutT from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Output columns n < n1 come from rows of W into C, columns n >= n1 from
// rows n - n1 of W2 into columns n - n1 of C2 (two projections of the same
// A in one launch; n1 = N for one).
template <typename InT, typename OutT, int MB>
__global__ void __launch_bounds__(kWarps * 32) skinny_gemm_kernel(
    const InT* __restrict__ A, long lda, const InT* __restrict__ W, long ldw,
    OutT* __restrict__ C, long ldc, const InT* __restrict__ W2, long ldw2,
    OutT* __restrict__ C2, long ldc2, int n1, int M, int N, int K) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = (blockIdx.x * kWarps + warp) * kRows;
  if (n0 >= N) return;
  const int nr = min(kRows, N - n0);
  const InT* wrow[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int n = n0 + r;
    wrow[r] = n < n1 ? W + static_cast<size_t>(n) * ldw : W2 + static_cast<size_t>(n - n1) * ldw2;
  }
  float acc[MB][kRows];
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int r = 0; r < kRows; ++r) acc[m][r] = 0.f;

  for (int k0 = lane * 8; k0 < K; k0 += 256 * kUnroll) {
    uint4 w[kUnroll][kRows];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int k = k0 + u * 256;
#pragma unroll
      for (int r = 0; r < kRows; ++r)
        w[u][r] = (k < K && r < nr) ? ld_stream(wrow[r] + k) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int k = k0 + u * 256;
      if (k < K) {
        float wf[kRows][8];
#pragma unroll
        for (int r = 0; r < kRows; ++r) to_f8<InT>(w[u][r], wf[r]);
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          if (m < M) {
            float af[8];
            to_f8<InT>(__ldg(reinterpret_cast<const uint4*>(A + static_cast<size_t>(m) * lda + k)),
                       af);
#pragma unroll
            for (int r = 0; r < kRows; ++r)
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[m][r] = fmaf(af[e], wf[r][e], acc[m][r]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MB; ++m) {
    if (m < M) {
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        float v = acc[m][r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0 && r < nr) {
          const int n = n0 + r;
          if (n < n1)
            C[static_cast<size_t>(m) * ldc + n] = from_f<OutT>(v);
          else
            C2[static_cast<size_t>(m) * ldc2 + (n - n1)] = from_f<OutT>(v);
        }
      }
    }
  }
}

template <typename InT, typename OutT>
cudaError_t launch_skinny_typed(const void* A, long lda, const void* W, long ldw, void* C,
                                long ldc, const void* W2, long ldw2, void* C2, long ldc2, int n1,
                                int M, int N, int K, cudaStream_t stream) {
  const int per_cta = kWarps * kRows;
  const dim3 grid((N + per_cta - 1) / per_cta);
  const InT* a = static_cast<const InT*>(A);
  const InT* w = static_cast<const InT*>(W);
  const InT* w2 = static_cast<const InT*>(W2);
  OutT* c = static_cast<OutT*>(C);
  OutT* c2 = static_cast<OutT*>(C2);
  const dim3 block(kWarps * 32);
  if (M <= 4)
    return launch_pdl(skinny_gemm_kernel<InT, OutT, 4>, grid, block, 0, stream, a, lda, w, ldw, c,
                      ldc, w2, ldw2, c2, ldc2, n1, M, N, K);
  if (M <= 8)
    return launch_pdl(skinny_gemm_kernel<InT, OutT, 8>, grid, block, 0, stream, a, lda, w, ldw, c,
                      ldc, w2, ldw2, c2, ldc2, n1, M, N, K);
  return launch_pdl(skinny_gemm_kernel<InT, OutT, 16>, grid, block, 0, stream, a, lda, w, ldw, c,
                    ldc, w2, ldw2, c2, ldc2, n1, M, N, K);
}

template <typename IT>
cudaError_t launch_skinny_out(const void* A, long lda, const void* W, long ldw, void* C, long ldc,
                              const void* W2, long ldw2, void* C2, long ldc2, int n1, int M, int N,
                              int K, int out_dtype, cudaStream_t stream) {
  switch (out_dtype) {
    case kF32:
      return launch_skinny_typed<IT, float>(A, lda, W, ldw, C, ldc, W2, ldw2, C2, ldc2, n1, M, N,
                                            K, stream);
    case kF16:
      return launch_skinny_typed<IT, __half>(A, lda, W, ldw, C, ldc, W2, ldw2, C2, ldc2, n1, M, N,
                                             K, stream);
    case kBF16:
      return launch_skinny_typed<IT, __nv_bfloat16>(A, lda, W, ldw, C, ldc, W2, ldw2, C2, ldc2,
                                                    n1, M, N, K, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_skinny_any(const void* A, long lda, const void* W, long ldw, void* C,
                              long ldc, const void* W2, long ldw2, void* C2, long ldc2, int n1,
                              int M, int N, int K, int in_dtype, int out_dtype,
                              cudaStream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
  if (M > kSkinnyMaxRows || K % 8 != 0) return cudaErrorInvalidValue;
  if (in_dtype == kBF16)
    return launch_skinny_out<__nv_bfloat16>(A, lda, W, ldw, C, ldc, W2, ldw2, C2, ldc2, n1, M, N,
                                            K, out_dtype, stream);
  if (in_dtype == kF16)
    return launch_skinny_out<__half>(A, lda, W, ldw, C, ldc, W2, ldw2, C2, ldc2, n1, M, N, K,
                                     out_dtype, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_linear_skinny(const void* A, long lda, const void* W, long ldw, void* C,
                                 long ldc, int M, int N, int K, int in_dtype, int out_dtype,
                                 cudaStream_t stream) {
  return launch_skinny_any(A, lda, W, ldw, C, ldc, W, ldw, C, ldc, N, M, N, K, in_dtype,
                           out_dtype, stream);
}

cudaError_t launch_linear_skinny2(const void* A, long lda, const void* W1, long ldw1, void* C1,
                                  long ldc1, int N1, const void* W2, long ldw2, void* C2,
                                  long ldc2, int N2, int M, int K, int in_dtype, int out_dtype,
                                  cudaStream_t stream) {
  return launch_skinny_any(A, lda, W1, ldw1, C1, ldc1, W2, ldw2, C2, ldc2, N1, M, N1 + N2, K,
                           in_dtype, out_dtype, stream);
}

}  // namespace g3
