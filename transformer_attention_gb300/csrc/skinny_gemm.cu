// C[M, N] = A[M, K] * W[N, K]^T for few rows (M <= 16): the projections of a
// decode step ("Gemma 3 Attention Block", How it works: Projections, with one
// new token per batch row).
//
// With M this small the product does 2*M flops per 2-byte weight, so it is
// bound by reading W once from HBM, and a 128-row tensor-core tile would be
// almost all padding.  Both kernels run on the CUDA cores with fp32 sums.
//
// skinny_bulk_kernel (rows of up to 10240 bf16): one persistent CTA per SM
// owns an even share of the output columns.  One elected thread streams
// its rows of W into a ring of shared-memory stages with bulk asynchronous
// copies (four rows per stage, up to 160 KB in flight per SM), issuing the
// first stages before it waits for the previous kernel; four groups of four
// consumer warps each reduce the rows of a stage (one row per warp) against
// the M rows of A (read through L1) and release the stage.  skinny_gemm_kernel (longer rows): each warp owns
// two rows of W and streams them with 16-byte loads, eight chunks of both
// rows in flight.
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

constexpr int kBulkConsumers = 4;                     // rows per stage = warps per group
constexpr int kBulkGroups = 4;                        // consumer groups (stages in work at once)
constexpr int kBulkThreads = 32 * (1 + kBulkConsumers * kBulkGroups);
constexpr int kBulkMaxStages = 8;
constexpr uint32_t kBulkRingBytes = 160 * 1024;       // shared memory for the ring

enum : int { kSiteBulkFull = 41, kSiteBulkEmpty = 42 };

// Output column n of this CTA's share [r0, r1) comes from row n of W (n < n1)
// or row n - n1 of W2.  `stages` ring stages of kBulkConsumers rows (K
// elements each) sit in dynamic shared memory; consumer group g < groups
// (warps 1 + 4g .. 4 + 4g) takes stages g, g + groups, ..., its warp c row c
// of each, so several stages are reduced at once (one warp per sub-partition
// could not hide the loads' latency).  `stages` is a multiple of `groups`:
// then every ring slot belongs to one group, which has consumed a slot's
// previous fill before it waits on the next one (an mbarrier parity wait
// cannot tell a phase from the one two fills earlier).
template <typename InT, typename OutT, int MB>
__global__ void __launch_bounds__(kBulkThreads, 1) skinny_bulk_kernel(
    const InT* __restrict__ A, long lda, const InT* __restrict__ W, long ldw,
    OutT* __restrict__ C, long ldc, const InT* __restrict__ W2, long ldw2,
    OutT* __restrict__ C2, long ldc2, int n1, int M, int N, int K, int stages, int groups,
    int* status) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[kBulkMaxStages], empty[kBulkMaxStages];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t row_bytes = static_cast<uint32_t>(K) * sizeof(InT);
  const uint32_t stage_bytes = row_bytes * kBulkConsumers;
  const int r0 = static_cast<int>(static_cast<long>(N) * blockIdx.x / gridDim.x);
  const int r1 = static_cast<int>(static_cast<long>(N) * (blockIdx.x + 1) / gridDim.x);
  const int nrows = r1 - r0;
  const int nst = (nrows + kBulkConsumers - 1) / kBulkConsumers;   // stages streamed
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kBulkConsumers);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- producer: this CTA's rows, kBulkConsumers per stage
      int fills[kBulkMaxStages] = {};
      bool waited = false;
      for (int s = 0; s < nst; ++s) {
        const int st = s % stages;
        if (s >= stages) {
          // The ring is full: from here on wait for the previous kernel too.
          if (!waited) {
            pdl_wait();
            pdl_trigger();
            waited = true;
          }
          if (!mbar_wait(smem_u32(&empty[st]), ((s / stages) - 1) & 1, &abort_flag, status,
                         kSiteBulkEmpty))
            break;
        }
        const int rows = min(kBulkConsumers, nrows - s * kBulkConsumers);
        const uint32_t fb = smem_u32(&full[st]);
        mbar_arrive_expect_tx(fb, rows * row_bytes);
        for (int i = 0; i < rows; ++i) {
          const int n = r0 + s * kBulkConsumers + i;
          const InT* src = n < n1 ? W + static_cast<size_t>(n) * ldw
                                  : W2 + static_cast<size_t>(n - n1) * ldw2;
          bulk_load(smem_u32(ring + st * stage_bytes + i * row_bytes), src, row_bytes, fb);
        }
        ++fills[st];
      }
      if (!waited) {
        pdl_wait();
        pdl_trigger();
      }
      // Every copy lands before shared memory is released.
      for (int i = 0; i < stages; ++i)
        if (fills[i] > 0) mbar_wait_drain(smem_u32(&full[i]), (fills[i] - 1) & 1);
    }
  } else {
    // ---------------- consumers: warp c of group g reduces row c of its stages
    pdl_enter();   // A is read and C written only after the previous kernel
    const int c = (warp - 1) % kBulkConsumers, g = (warp - 1) / kBulkConsumers;
    for (int s = g; g < groups && s < nst; s += groups) {
      const int st = s % stages;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[st]), (s / stages) & 1, &abort_flag,
                                             status, kSiteBulkFull)))
        break;
      const int r = s * kBulkConsumers + c;
      if (r < nrows) {
        const InT* wr = reinterpret_cast<const InT*>(ring + st * stage_bytes + c * row_bytes);
        float acc[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) acc[m] = 0.f;
#pragma unroll 2
        for (int k = lane * 8; k < K; k += 256) {
          float wf[8];
          to_f8<InT>(*reinterpret_cast<const uint4*>(wr + k), wf);
#pragma unroll
          for (int m = 0; m < MB; ++m) {
            if (m < M) {
              float af[8];
              to_f8<InT>(
                  __ldg(reinterpret_cast<const uint4*>(A + static_cast<size_t>(m) * lda + k)), af);
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[m] = fmaf(af[e], wf[e], acc[m]);
            }
          }
        }
        const int n = r0 + r;
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          if (m < M) {
            float v = acc[m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) {
              if (n < n1)
                C[static_cast<size_t>(m) * ldc + n] = from_f<OutT>(v);
              else
                C2[static_cast<size_t>(m) * ldc2 + (n - n1)] = from_f<OutT>(v);
            }
          }
        }
      }
      // This warp's reads of the stage are done: the producer may refill it.
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
    }
  }
}

// Ring stages for rows of K elements: the largest of 2, 4, 8 that fits in
// kBulkRingBytes, or 0 when two do not fit or the rows cannot be
// bulk-copied (16-byte alignment of the weights and their row strides).
template <typename InT>
int bulk_stages(const void* W, long ldw, const void* W2, long ldw2, int K) {
  const uint64_t row_bytes = static_cast<uint64_t>(K) * sizeof(InT);
  const auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (row_bytes % 16 != 0 || !al(W) || !al(W2) || (ldw * sizeof(InT)) % 16 != 0 ||
      (ldw2 * sizeof(InT)) % 16 != 0)
    return 0;
  const uint64_t st = kBulkRingBytes / (row_bytes * kBulkConsumers);
  return st >= 8 ? 8 : st >= 4 ? 4 : st >= 2 ? 2 : 0;
}

template <typename InT, typename OutT, int MB>
cudaError_t launch_bulk(const InT* a, long lda, const InT* w, long ldw, OutT* c, long ldc,
                        const InT* w2, long ldw2, OutT* c2, long ldc2, int n1, int M, int N,
                        int K, int stages, cudaStream_t stream, int* status) {
  auto kern = skinny_bulk_kernel<InT, OutT, MB>;
  static bool attr_set = false;  // benign race: setting the same attribute twice is harmless
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kBulkRingBytes));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const size_t smem = static_cast<size_t>(stages) * K * sizeof(InT) * kBulkConsumers;
  const int grid = N < num_sms() ? N : num_sms();
  const int groups = stages < kBulkGroups ? stages : kBulkGroups;   // divides stages
  return launch_pdl(kern, dim3(grid), dim3(kBulkThreads), smem, stream, a, lda, w, ldw, c, ldc,
                    w2, ldw2, c2, ldc2, n1, M, N, K, stages, groups, status);
}

template <typename InT, typename OutT>
cudaError_t launch_skinny_typed(const void* A, long lda, const void* W, long ldw, void* C,
                                long ldc, const void* W2, long ldw2, void* C2, long ldc2, int n1,
                                int M, int N, int K, cudaStream_t stream, int* status) {
  const int stages = bulk_stages<InT>(W, ldw, W2, ldw2, K);
  if (stages > 0) {
    const InT* a = static_cast<const InT*>(A);
    const InT* w = static_cast<const InT*>(W);
    const InT* w2 = static_cast<const InT*>(W2);
    OutT* c = static_cast<OutT*>(C);
    OutT* c2 = static_cast<OutT*>(C2);
    if (M <= 1)
      return launch_bulk<InT, OutT, 1>(a, lda, w, ldw, c, ldc, w2, ldw2, c2, ldc2, n1, M, N, K,
                                       stages, stream, status);
    if (M <= 2)
      return launch_bulk<InT, OutT, 2>(a, lda, w, ldw, c, ldc, w2, ldw2, c2, ldc2, n1, M, N, K,
                                       stages, stream, status);
    if (M <= 4)
      return launch_bulk<InT, OutT, 4>(a, lda, w, ldw, c, ldc, w2, ldw2, c2, ldc2, n1, M, N, K,
                                       stages, stream, status);
    if (M <= 8)
      return launch_bulk<InT, OutT, 8>(a, lda, w, ldw, c, ldc, w2, ldw2, c2, ldc2, n1, M, N, K,
                                       stages, stream, status);
    return launch_bulk<InT, OutT, 16>(a, lda, w, ldw, c, ldc, w2, ldw2, c2, ldc2, n1, M, N, K,
                                      stages, stream, status);
  }
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
                              int K, int out_dtype, cudaStream_t stream, int* status) {
  switch (out_dtype) {
    case kF32:
      return launch_skinny_typed<IT, float>(A, lda, W, ldw, C, ldc, W2, ldw2, C2, ldc2, n1, M, N,
                                            K, stream, status);
    case kF16:
      return launch_skinny_typed<IT, __half>(A, lda, W, ldw, C, ldc, W2, ldw2, C2, ldc2, n1, M, N,
                                             K, stream, status);
    case kBF16:
      return launch_skinny_typed<IT, __nv_bfloat16>(A, lda, W, ldw, C, ldc, W2, ldw2, C2, ldc2,
                                                    n1, M, N, K, stream, status);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_skinny_any(const void* A, long lda, const void* W, long ldw, void* C,
                              long ldc, const void* W2, long ldw2, void* C2, long ldc2, int n1,
                              int M, int N, int K, int in_dtype, int out_dtype,
                              cudaStream_t stream, int* status) {
  if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
  if (M > kSkinnyMaxRows || K % 8 != 0) return cudaErrorInvalidValue;
  if (in_dtype == kBF16)
    return launch_skinny_out<__nv_bfloat16>(A, lda, W, ldw, C, ldc, W2, ldw2, C2, ldc2, n1, M, N,
                                            K, out_dtype, stream, status);
  if (in_dtype == kF16)
    return launch_skinny_out<__half>(A, lda, W, ldw, C, ldc, W2, ldw2, C2, ldc2, n1, M, N, K,
                                     out_dtype, stream, status);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_linear_skinny(const void* A, long lda, const void* W, long ldw, void* C,
                                 long ldc, int M, int N, int K, int in_dtype, int out_dtype,
                                 cudaStream_t stream, int* status) {
  return launch_skinny_any(A, lda, W, ldw, C, ldc, W, ldw, C, ldc, N, M, N, K, in_dtype,
                           out_dtype, stream, status);
}

cudaError_t launch_linear_skinny2(const void* A, long lda, const void* W1, long ldw1, void* C1,
                                  long ldc1, int N1, const void* W2, long ldw2, void* C2,
                                  long ldc2, int N2, int M, int K, int in_dtype, int out_dtype,
                                  cudaStream_t stream, int* status) {
  return launch_skinny_any(A, lda, W1, ldw1, C1, ldc1, W2, ldw2, C2, ldc2, N1, M, N1 + N2, K,
                           in_dtype, out_dtype, stream, status);
}

}  // namespace g3
