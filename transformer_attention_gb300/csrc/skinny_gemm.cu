// C[M, N] = A[M, K] * W[N, K]^T for few rows (M <= 16): the projections of a
// decode step ("Gemma 3 Attention Block", How it works: Projections, with one
// new token per batch row).
//
// With M this small the product does 2*M flops per 2-byte weight, so it is
// bound by reading W once from HBM.  The tensor cores still do the
// arithmetic, with the operands' roles swapped so that the weights fill the
// 128-row side of the MMA: D[128 rows of W, 16] = W_tile A^T (tcgen05,
// M = 128, N = 16; the rows of A past M are read as zeros by TMA).  The CUDA
// cores then execute no per-element instructions and the kernel is a TMA
// stream of W.  A tile of 128 rows of W has K/64 k-blocks; to put enough
// CTAs on the GPU the k-blocks of a tile are split over a cluster of up to 8
// CTAs, and the cluster's rank-0 CTA sums their fp32 partials through
// distributed shared memory before it writes C.
//
// One CTA (4 warps, two CTAs per SM): warp 0's elected lane streams W boxes
// {64 k, 128 rows} and A boxes {64 k, 16 rows} (128-byte swizzle) into a
// 4-stage ring, issuing the W copies of the first stages before it waits for
// the previous kernel (no kernel of the library writes weights, and only the
// library's kernels let the next kernel start early); warp 1 allocates 32
// TMEM columns and issues the MMAs; then all four warps read the
// accumulator (warp w: rows 32w .. 32w + 31 of the tile).  Every mbarrier
// wait is bounded (ptx.cuh).
#include "internal.h"
#include "ptx.cuh"

namespace g3 {

namespace {

constexpr int TN = 128;   // rows of W per tile (the MMA's M)
constexpr int MA = 16;    // rows of A per MMA (the MMA's N); M <= 16
constexpr int KB = 64;    // k per block
constexpr int STAGES = 4;
constexpr int CTAS_PER_SM = 2;
constexpr int THREADS = 128;
constexpr int MAX_SPLITS = 8;   // portable cluster size
constexpr uint32_t W_BYTES = TN * KB * 2;                 // 16 KB
constexpr uint32_t A_BYTES = MA * KB * 2;                 // 2 KB
constexpr uint32_t STAGE_BYTES = W_BYTES + A_BYTES;       // 18 KB, a multiple of 1 KB
constexpr uint32_t RED_BYTES = TN * MA * 4;               // fp32 partials of the tile
constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + RED_BYTES + 1024;
constexpr uint32_t TMEM_COLS = 32;                        // the smallest allocation

enum : int { kSiteSkFull = 41, kSiteSkEmpty = 42, kSiteSkDone = 43 };

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

// Output column n comes from row n of W (tmW, n < n1) or row n - n1 of W2
// (tmW2) and goes to C or to column n - n1 of C2; n1 is a multiple of TN.
// CTA b works on tile b / splits, k-block share b % splits (its rank in a
// cluster of `splits` CTAs).
template <int AB_BF16, typename OutT>
__global__ void __launch_bounds__(THREADS, CTAS_PER_SM)
    skinny_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW2,
                     const __grid_constant__ CUtensorMap tmA, OutT* __restrict__ C, long ldc,
                     OutT* __restrict__ C2, long ldc2, int n1, int M, int N, int K, int splits,
                     int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  float* red = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES);
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], done;
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_flag;
  __shared__ int partial_ok;   // 0 once a warp of this CTA found its MMAs unfinished
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / splits, split = blockIdx.x % splits;
  const int row0 = tile * TN;
  const bool seg2 = row0 >= n1;
  const CUtensorMap* wmap = seg2 ? &tmW2 : &tmW;
  const int wrow = seg2 ? row0 - n1 : row0;
  const int nkb = (K + KB - 1) / KB;
  const int kb0 = nkb * split / splits;
  const int nk = nkb * (split + 1) / splits - kb0;   // >= 1: splits <= nkb

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(&done), 1);
    abort_flag = 0;
    partial_ok = 1;
    fence_barrier_init();
    tma_prefetch_desc(wmap);
    tma_prefetch_desc(&tmA);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_sh), TMEM_COLS);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_sh;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- producer
      const int pre = nk < STAGES ? nk : STAGES;
      int fills[STAGES] = {};
      for (int j = 0; j < pre; ++j) {   // weights only: no earlier kernel writes them
        const uint32_t fb = smem_u32(&full[j]);
        mbar_arrive_expect_tx(fb, STAGE_BYTES);
        tma_load_2d(smem_u32(smem + j * STAGE_BYTES), wmap, fb, (kb0 + j) * KB, wrow);
        fills[j] = 1;
      }
      pdl_wait();
      pdl_trigger();
      for (int j = 0; j < pre; ++j)
        tma_load_2d(smem_u32(smem + j * STAGE_BYTES + W_BYTES), &tmA, smem_u32(&full[j]),
                    (kb0 + j) * KB, 0);
      for (int j = pre; j < nk; ++j) {
        const int st = j % STAGES;
        if (!mbar_wait(smem_u32(&empty[st]), ((j / STAGES) - 1) & 1, &abort_flag, status,
                       kSiteSkEmpty))
          break;
        const uint32_t fb = smem_u32(&full[st]);
        mbar_arrive_expect_tx(fb, STAGE_BYTES);
        tma_load_2d(smem_u32(smem + st * STAGE_BYTES), wmap, fb, (kb0 + j) * KB, wrow);
        tma_load_2d(smem_u32(smem + st * STAGE_BYTES + W_BYTES), &tmA, fb, (kb0 + j) * KB, 0);
        ++fills[st];
      }
      // Every copy lands before shared memory is released.
      for (int s = 0; s < STAGES; ++s)
        if (fills[s] > 0) mbar_wait_drain(smem_u32(&full[s]), (fills[s] - 1) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer: the whole warp runs the loop, one elected
    // lane issues each tcgen05 instruction
    const uint32_t lead = elect_one();
    constexpr uint32_t idesc = idesc_f16(TN, MA, AB_BF16, 0, 0);
    for (int j = 0; j < nk; ++j) {
      const int st = j % STAGES;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[st]), (j / STAGES) & 1, &abort_flag,
                                             status, kSiteSkFull)))
        break;
      tc_fence_after();
      const uint32_t w_addr = smem_u32(smem + st * STAGE_BYTES);
      const uint32_t a_addr = w_addr + W_BYTES;
#pragma unroll
      for (int k = 0; k < KB / 16; ++k)
        mma_ss_lead(lead, tbase, sdesc_sw128(w_addr + k * 32, 16, 1024),
                    sdesc_sw128(a_addr + k * 32, 16, 1024), idesc, (j | k) != 0 ? 1u : 0u);
      mma_commit_lead(lead, smem_u32(&empty[st]));
    }
    // After the MMAs issued so far (all of them unless a wait gave up).
    mma_commit_lead(lead, smem_u32(&done));
  }

  // ---------------- epilogue: all four warps, row r of the tile per thread
  pdl_wait();   // C is written only after the previous kernel
  pdl_trigger();
  bool got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&done), 0, &abort_flag, status,
                                               kSiteSkDone));
  tc_fence_after();
  uint32_t v[32];   // columns 0 .. MA - 1 hold this row's products with the rows of A
  tmem_ld32(tbase + (static_cast<uint32_t>(warp * 32) << 16), v);
  tmem_ld_wait(v);
  const int r = warp * 32 + lane;
  if (splits > 1) {
#pragma unroll
    for (int m = 0; m < MA; ++m)
      if (m < M) red[r * MA + m] = __uint_as_float(v[m]);
    if (!got && lane == 0) partial_ok = 0;
    cluster_sync();   // every CTA's partials and flag are in its shared memory
    if (split == 0) {
      // a peer whose MMAs did not all complete holds a stale partial: no store
      got = partial_ok != 0;
      for (int q = 1; q < splits; ++q)
        got = got && ld_shared_cluster_u32(mapa_shared(smem_u32(&partial_ok),
                                                       static_cast<uint32_t>(q))) != 0;
      for (int q = 1; q < splits; ++q) {
        const uint32_t peer = mapa_shared(smem_u32(red + r * MA), static_cast<uint32_t>(q));
#pragma unroll
        for (int m = 0; m < MA; ++m)
          if (m < M)
            v[m] = __float_as_uint(__uint_as_float(v[m]) + ld_shared_cluster_f32(peer + m * 4));
      }
    }
  }
  const int n = row0 + r;
  if (split == 0 && got && n < N) {
#pragma unroll
    for (int m = 0; m < MA; ++m) {
      if (m < M) {
        if (n < n1)
          C[static_cast<size_t>(m) * ldc + n] = from_f<OutT>(__uint_as_float(v[m]));
        else
          C2[static_cast<size_t>(m) * ldc2 + (n - n1)] = from_f<OutT>(__uint_as_float(v[m]));
      }
    }
  }
  if (splits > 1) cluster_sync();   // rank 0 has read the peers' partials
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

// Tensor maps over W (rows of K elements, row stride ldw) and A, boxes of 64
// k by `rows` rows, 128-byte swizzle.
bool encode_rows(CUtensorMap& map, const void* base, long ld, int K, int rows_total,
                 uint32_t box_rows, int in_dtype) {
  const CUtensorMapDataType dt =
      in_dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows_total)};
  const uint64_t str[1] = {static_cast<uint64_t>(ld) * 2};
  const uint32_t box[2] = {static_cast<uint32_t>(KB), box_rows};
  return encode_tiled(&map, dt, 2, base, dims, str, box);
}

template <int AB, typename OutT>
cudaError_t launch_tc(const CUtensorMap& tw, const CUtensorMap& tw2, const CUtensorMap& ta,
                      void* C, long ldc, void* C2, long ldc2, int n1, int M, int N, int K,
                      cudaStream_t stream, int* status) {
  auto kern = skinny_tc_kernel<AB, OutT>;
  if (cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), SMEM_BYTES))
    return e;
  // Split each tile's k-blocks over enough CTAs to fill every SM.
  const int tiles = (N + TN - 1) / TN;
  const int nkb = (K + KB - 1) / KB;
  int splits = CTAS_PER_SM * num_sms() / tiles;
  if (splits > MAX_SPLITS) splits = MAX_SPLITS;
  if (splits > nkb) splits = nkb;
  if (splits < 1) splits = 1;
  OutT* c = static_cast<OutT*>(C);
  OutT* c2 = static_cast<OutT*>(C2);
  const dim3 grid(tiles * splits);
  if (splits == 1)
    return launch_pdl(kern, grid, dim3(THREADS), SMEM_BYTES, stream, tw, tw2, ta, c, ldc, c2,
                      ldc2, n1, M, N, K, splits, status);
  return launch_pdl_cluster(kern, grid, dim3(THREADS), SMEM_BYTES, splits, stream, tw, tw2, ta, c,
                            ldc, c2, ldc2, n1, M, N, K, splits, status);
}

// One launch over the columns [0, N) (two weight segments split at n1, a
// multiple of TN, or n1 = N).
cudaError_t launch_segments(const void* A, long lda, const void* W, long ldw, void* C, long ldc,
                            const void* W2, long ldw2, void* C2, long ldc2, int n1, int M, int N,
                            int K, int in_dtype, int out_dtype, cudaStream_t stream, int* status) {
  CUtensorMap tw, tw2, ta;
  if (!encode_rows(tw, W, ldw, K, n1, TN, in_dtype) ||
      !encode_rows(ta, A, lda, K, M, MA, in_dtype))
    return cudaErrorInvalidValue;
  tw2 = tw;
  if (n1 < N && !encode_rows(tw2, W2, ldw2, K, N - n1, TN, in_dtype)) return cudaErrorInvalidValue;
#define G3_SK_OUT(AB)                                                                            \
  switch (out_dtype) {                                                                           \
    case kF32:                                                                                   \
      return launch_tc<AB, float>(tw, tw2, ta, C, ldc, C2, ldc2, n1, M, N, K, stream, status);   \
    case kF16:                                                                                   \
      return launch_tc<AB, __half>(tw, tw2, ta, C, ldc, C2, ldc2, n1, M, N, K, stream, status);  \
    case kBF16:                                                                                  \
      return launch_tc<AB, __nv_bfloat16>(tw, tw2, ta, C, ldc, C2, ldc2, n1, M, N, K, stream,    \
                                          status);                                               \
    default: return cudaErrorInvalidValue;                                                       \
  }
  if (in_dtype == kBF16) {
    G3_SK_OUT(1)
  }
  G3_SK_OUT(0)
#undef G3_SK_OUT
}

cudaError_t launch_skinny_any(const void* A, long lda, const void* W, long ldw, void* C,
                              long ldc, const void* W2, long ldw2, void* C2, long ldc2, int n1,
                              int M, int N, int K, int in_dtype, int out_dtype,
                              cudaStream_t stream, int* status) {
  if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
  if (M > kSkinnyMaxRows || K % 8 != 0) return cudaErrorInvalidValue;
  if (in_dtype != kBF16 && in_dtype != kF16) return cudaErrorInvalidValue;
  // (the two-segment callers split at H * d_h, a multiple of TN)
  if (n1 < N && n1 % TN != 0) return cudaErrorInvalidValue;
  return launch_segments(A, lda, W, ldw, C, ldc, W2, ldw2, C2, ldc2, n1 < N ? n1 : N, M, N, K,
                         in_dtype, out_dtype, stream, status);
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
