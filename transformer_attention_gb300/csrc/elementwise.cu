// Memory-bound kernels of the attention block.
//
// qk_norm_rope: the fused prologue between the projections and attention
//   ("QK-Norm", How it works; "Gemma 3 Attention Block", How it works:
//   QK-norm, then RoPE, then scale).  For every token and every query / key
//   head vector x in R^{d_h}:
//     x <- x / sqrt(mean(x^2) + 1e-6) * (1 + gamma)     (gamma_q or gamma_k)
//     x <- RoPE(x; pos, base, scale)                     (pairs (c, c + d_h/2),
//          angle (pos / scale) * base^(-2c/d_h))
//     Q only: x <- x * query_scale
//   One warp per token, d_h/8 lanes per head vector, 8 fp16 elements (one
//   16-byte load) per lane; the RMS is a shuffle reduction over those lanes
//   and the RoPE partner element sits d_h/16 lanes away.  Angles: rope.cuh.
//   Rows are updated in place.  (The layer pipelines fuse this step into the
//   projection GEMM's epilogue; this kernel serves the cases that fusion does
//   not cover and the stage entry point.)
//
// embed_rows: the model's input ("Full Gemma 3 Block", How it works, last
//   paragraph: embed times sqrt(D)), x[m, :] = E[tokens[m], :] * scale in fp32.
//
// rmsnorm_rows / postnorm_residual: the D-axis norms of the block sandwich
//   ("Full Gemma 3 Block", How it works: a = Attn(RMSNorm_pre(x));
//   a <- RMSNorm_post(a); h = x + a), one warp per row.
#include <cmath>

#include "decode_span.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace g3 {

namespace {

constexpr float kEps = 1e-6f;

constexpr int kVecUnroll = 8;  // head vectors in flight per lane

// Work items are (row m, chunk of up to chunk_u * VPW head vectors): a warp
// per item, so that a decode step's few rows spread over many warps
// (chunk_u = 1) while long inputs amortise the angle math over a row's
// vectors (chunk_u = kVecUnroll).
template <int DH>
__global__ void __launch_bounds__(256, 2)
    qk_norm_rope_kernel(__half* __restrict__ Q, long ldq, __half* __restrict__ K, long ldk,
                        const __nv_bfloat16* __restrict__ gamma_q,
                        const __nv_bfloat16* __restrict__ gamma_k, const int32_t* __restrict__ pos,
                        int M, int H, int H_kv, const __grid_constant__ RopeFreqs freqs,
                        float query_scale, const __grid_constant__ CacheRows cache, int chunk_u,
                        int qk_blocks) {
  pdl_enter();
  if (static_cast<int>(blockIdx.x) >= qk_blocks) {
    // CTAs past qk_blocks scan the local layer's cache span for the cache
    // attention of a decode step: CTA qk_blocks + b * nchunk + c takes chunk c
    // of row b.
    const int idx = static_cast<int>(blockIdx.x) - qk_blocks;
    kv_span_chunk(cache.posc, pos, cache.pad_lens, cache.T, cache.S, cache.end, cache.window,
                  cache.nchunk, cache.span_part, idx % cache.nchunk, idx / cache.nchunk);
    return;
  }
  constexpr int LPV = DH / 8;      // lanes per head vector
  constexpr int VPW = 32 / LPV;    // head vectors per warp step
  constexpr int HALF = LPV / 2;    // lane distance of the RoPE partner
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPV, ll = lane % LPV;
  const bool second_half = ll >= HALF;
  const int c0 = (ll % HALF) * 8;  // first rotation pair index of this lane

  // (1 + gamma) of this lane's 8 channels, kept packed (bf16x8) to save registers.
  const uint4 gq_raw = *reinterpret_cast<const uint4*>(gamma_q + ll * 8);
  const uint4 gk_raw = *reinterpret_cast<const uint4*>(gamma_k + ll * 8);

  const int warps_total = qk_blocks * (blockDim.x >> 5);
  const int nvec = H + H_kv;
  const int vpc = VPW * chunk_u;                   // head vectors per item
  const int nch = (nvec + vpc - 1) / vpc;          // items per row
  const long items = static_cast<long>(M) * nch;
  const int KVD = H_kv * DH;
  __half* const Kc = static_cast<__half*>(cache.Kc);
  for (long item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < items;
       item += warps_total) {
    const int m = static_cast<int>(item / nch);
    const int base = static_cast<int>(item % nch) * vpc;   // first head vector of the item
    // this row's cache slot (with cache.Kc)
    const size_t slot =
        static_cast<size_t>(m / cache.T) * cache.S + cache.end + m % cache.T;
    // Issue the item's head-vector loads first, then the angle math.
    uint4 raw[kVecUnroll];
    const int first = base + sub;
#pragma unroll
    for (int u = 0; u < kVecUnroll; ++u) {
      const int hv = first + u * VPW;
      const __half* src = hv < H ? Q + static_cast<long>(m) * ldq + hv * DH
                                 : K + static_cast<long>(m) * ldk + (hv - H) * DH;
      raw[u] = (u < chunk_u && hv < nvec) ? *reinterpret_cast<const uint4*>(src + ll * 8)
                                          : make_uint4(0, 0, 0, 0);
    }
    const float p = static_cast<float>(pos[m]);
    float cs[8], sn[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) rope_sincos(p, freqs.f[c0 + e], sn[e], cs[e]);
    {
#pragma unroll
      for (int u = 0; u < kVecUnroll; ++u) {
        if (u >= chunk_u || base + u * VPW >= nvec) break;   // warp-uniform
        const int hv = first + u * VPW;
        const bool is_q = hv < H;
        float x[8];
        const __half2* h2 = reinterpret_cast<const __half2*>(&raw[u]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(h2[e]);
          x[2 * e] = f.x;
          x[2 * e + 1] = f.y;
        }
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
        for (int off = HALF; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float rs = rsqrtf(ss * (1.f / DH) + kEps);
        const uint4 graw = is_q ? gq_raw : gk_raw;
        const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&graw);
        float y[8], o[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 gf = __bfloat1622float2(g2[e]);
          y[2 * e] = x[2 * e] * rs * (1.f + gf.x);
          y[2 * e + 1] = x[2 * e + 1] * rs * (1.f + gf.y);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = __shfl_xor_sync(0xffffffffu, y[e], HALF);
        const float sc = is_q ? query_scale : 1.f;
        uint4 w;
        uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float r0, r1;
          if (!second_half) {  // y is x1 (first half), o is x2
            r0 = y[2 * e] * cs[2 * e] - o[2 * e] * sn[2 * e];
            r1 = y[2 * e + 1] * cs[2 * e + 1] - o[2 * e + 1] * sn[2 * e + 1];
          } else {             // y is x2, o is x1
            r0 = y[2 * e] * cs[2 * e] + o[2 * e] * sn[2 * e];
            r1 = y[2 * e + 1] * cs[2 * e + 1] + o[2 * e + 1] * sn[2 * e + 1];
          }
          wp[e] = pack_half2(r0 * sc, r1 * sc);
        }
        if (hv < nvec) {
          __half* dst = is_q ? Q + static_cast<long>(m) * ldq + hv * DH
                             : K + static_cast<long>(m) * ldk + (hv - H) * DH;
          *reinterpret_cast<uint4*>(dst + ll * 8) = w;
          if (!is_q && Kc != nullptr) {
            // K' head j and V head j of the row go to its cache slot
            const int off = (hv - H) * DH + ll * 8;
            *reinterpret_cast<uint4*>(Kc + slot * KVD + off) = w;
            *reinterpret_cast<uint4*>(static_cast<__half*>(cache.Vc) + slot * KVD + off) =
                *reinterpret_cast<const uint4*>(static_cast<const __half*>(cache.V) +
                                                static_cast<long>(m) * cache.ldv + off);
          }
        }
      }
    }
    if (Kc != nullptr && base == 0 && lane == 0) {   // the slot's position
      const int b = m / cache.T, t = m % cache.T;
      const int valid = cache.T - (cache.pad_lens != nullptr ? cache.pad_lens[b] : 0);
      cache.posc[slot] = t < valid ? pos[m] : -1;
    }
  }
}

template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <> __device__ __forceinline__ float4 load4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <> __device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// Row m lies past its segment's valid length.
__device__ __forceinline__ bool pad_row(const PadRows& p, int m) {
  if (p.pad_lens == nullptr) return false;
  const int b = m / p.seg_T, t = m - b * p.seg_T;
  return t >= p.seg_T - p.pad_lens[b];
}

// Row m lies in a 128-row tile of its segment holding pad rows only (a tile
// the projection GEMMs neither read nor compute).
__device__ __forceinline__ bool pad_tile_row(const PadRows& p, int m) {
  if (p.pad_lens == nullptr || p.seg_T % 128 != 0) return false;
  const int b = m / p.seg_T, t = m - b * p.seg_T;
  return (t & ~127) >= p.seg_T - p.pad_lens[b];
}

// u = RMSNorm(x) * (1 + gamma) -> bf16 or fp16, one warp per row, D % 4 == 0.
template <typename T, bool OUT_F16>
__global__ void __launch_bounds__(256)
    rmsnorm_rows_kernel(const T* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
                        uint16_t* __restrict__ u, int M, int D, PadRows pad) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= M || pad_tile_row(pad, row)) return;
  const T* xr = x + static_cast<long>(row) * D;
  float ss = 0.f;
  for (int c = lane * 4; c < D; c += 128) {
    const float4 v = load4<T>(xr + c);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float rs = rsqrtf(ss / D + kEps);
  uint16_t* ur = u + static_cast<long>(row) * D;
  for (int c = lane * 4; c < D; c += 128) {
    const float4 v = load4<T>(xr + c);
    const float4 g = load4<__nv_bfloat16>(gamma + c);
    const float a0 = v.x * rs * (1.f + g.x), a1 = v.y * rs * (1.f + g.y);
    const float a2 = v.z * rs * (1.f + g.z), a3 = v.w * rs * (1.f + g.w);
    uint2 w;
    if (OUT_F16) {
      w.x = pack_half2(a0, a1);
      w.y = pack_half2(a2, a3);
    } else {
      w.x = pack_bf162(a0, a1);
      w.y = pack_bf162(a2, a3);
    }
    *reinterpret_cast<uint2*>(ur + c) = w;
  }
}

// The same with the row held in registers (NV 4-element vectors per lane,
// D <= 128 * NV): every load of the row is issued before the sum, and x is
// read once.
template <typename T, bool OUT_F16, int NV>
__global__ void __launch_bounds__(128)
    rmsnorm_rows_reg_kernel(const T* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
                            uint16_t* __restrict__ u, int M, int D, PadRows pad) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= M || pad_tile_row(pad, row)) return;
  const T* xr = x + static_cast<long>(row) * D;
  float4 v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = lane * 4 + i * 128;
    v[i] = c < D ? load4<T>(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i)
    ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float rs = rsqrtf(ss / D + kEps);
  uint16_t* ur = u + static_cast<long>(row) * D;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = lane * 4 + i * 128;
    if (c < D) {
      const float4 g = load4<__nv_bfloat16>(gamma + c);
      const float a0 = v[i].x * rs * (1.f + g.x), a1 = v[i].y * rs * (1.f + g.y);
      const float a2 = v[i].z * rs * (1.f + g.z), a3 = v[i].w * rs * (1.f + g.w);
      uint2 w;
      if (OUT_F16) {
        w.x = pack_half2(a0, a1);
        w.y = pack_half2(a2, a3);
      } else {
        w.x = pack_bf162(a0, a1);
        w.y = pack_bf162(a2, a3);
      }
      *reinterpret_cast<uint2*>(ur + c) = w;
    }
  }
}

// bf16 -> fp16, 8 elements per thread per step (n % 8 == 0, 16-byte aligned).
__global__ void __launch_bounds__(256)
    cast_bf16_f16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n8) {
  pdl_enter();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 v = src[i];
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&in[e]));
      out[e] = pack_half2(f.x, f.y);
    }
    dst[i] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// A pad row's y = x + RMSNorm(0) = x: copied (as fp32) unless y is x.
template <typename T>
__device__ __forceinline__ void pad_row_residual(const T* x, float* y, int row, int D, int lane,
                                                 int inplace) {
  if (inplace) return;
  const T* xr = x + static_cast<long>(row) * D;
  float* yr = y + static_cast<long>(row) * D;
  for (int c = lane * 4; c < D; c += 128) *reinterpret_cast<float4*>(yr + c) = load4<T>(xr + c);
}

// y = x + RMSNorm(a) * (1 + gamma), one warp per row; y may alias x (f32).
template <typename T>
__global__ void __launch_bounds__(256)
    postnorm_residual_kernel(const float* __restrict__ a, const T* x,
                             const __nv_bfloat16* __restrict__ gamma, float* y, int M, int D,
                             PadRows pad, int inplace) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= M) return;
  if (pad_row(pad, row)) {
    pad_row_residual(x, y, row, D, lane, inplace);
    return;
  }
  const float* ar = a + static_cast<long>(row) * D;
  float ss = 0.f;
  for (int c = lane * 4; c < D; c += 128) {
    const float4 v = *reinterpret_cast<const float4*>(ar + c);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float rs = rsqrtf(ss / D + kEps);
  const T* xr = x + static_cast<long>(row) * D;
  float* yr = y + static_cast<long>(row) * D;
  for (int c = lane * 4; c < D; c += 128) {
    const float4 v = *reinterpret_cast<const float4*>(ar + c);
    const float4 g = load4<__nv_bfloat16>(gamma + c);
    const float4 xv = load4<T>(xr + c);
    float4 o;
    o.x = xv.x + v.x * rs * (1.f + g.x);
    o.y = xv.y + v.y * rs * (1.f + g.y);
    o.z = xv.z + v.z * rs * (1.f + g.z);
    o.w = xv.w + v.w * rs * (1.f + g.w);
    *reinterpret_cast<float4*>(yr + c) = o;
  }
}

// The same with a's row held in registers (D <= 128 * NV): a is read once.
template <typename T, int NV>
__global__ void __launch_bounds__(128)
    postnorm_residual_reg_kernel(const float* __restrict__ a, const T* x,
                                 const __nv_bfloat16* __restrict__ gamma, float* y, int M, int D,
                                 PadRows pad, int inplace) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= M) return;
  if (pad_row(pad, row)) {
    pad_row_residual(x, y, row, D, lane, inplace);
    return;
  }
  const float* ar = a + static_cast<long>(row) * D;
  float4 v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = lane * 4 + i * 128;
    v[i] = c < D ? *reinterpret_cast<const float4*>(ar + c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i)
    ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float rs = rsqrtf(ss / D + kEps);
  const T* xr = x + static_cast<long>(row) * D;
  float* yr = y + static_cast<long>(row) * D;
  // y may alias x, so x is loaded eight vectors at a time before their stores
  // (a batch of loads in flight instead of one load per store).
#pragma unroll
  for (int i0 = 0; i0 < NV; i0 += 8) {
    float4 xv[8], g[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = lane * 4 + (i0 + j) * 128;
      if (c < D) {
        xv[j] = load4<T>(xr + c);
        g[j] = load4<__nv_bfloat16>(gamma + c);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = lane * 4 + (i0 + j) * 128;
      if (c < D) {
        const float4& a4 = v[i0 + j];
        float4 o;
        o.x = xv[j].x + a4.x * rs * (1.f + g[j].x);
        o.y = xv[j].y + a4.y * rs * (1.f + g[j].y);
        o.z = xv[j].z + a4.z * rs * (1.f + g[j].z);
        o.w = xv[j].w + a4.w * rs * (1.f + g[j].w);
        *reinterpret_cast<float4*>(yr + c) = o;
      }
    }
  }
}

// Row widths 2049..4096 (and up to 6144 for the pre-norm) are read once,
// from registers, one warp per row and 4 rows per CTA (their 150-250
// registers per thread would otherwise leave one CTA per SM).  Narrower
// rows use the two-pass kernels (8 rows per CTA): their second pass finds
// the row still in cache, and their low register use keeps more rows in
// flight.  At 48 vectors per lane the post-norm's row and batch of x would
// not fit in registers, so those widths use its two-pass kernel too.
inline dim3 row_grid(int M, int rows) { return dim3((M + rows - 1) / rows); }

template <typename T, bool OUT_F16>
cudaError_t launch_rms_typed(cudaStream_t s, const T* x, const __nv_bfloat16* g, uint16_t* u,
                             int M, int D, const PadRows& pad) {
  if (D > 2048 && D <= 4096)
    return launch_pdl(rmsnorm_rows_reg_kernel<T, OUT_F16, 32>, row_grid(M, 4), dim3(128), 0, s,
                      x, g, u, M, D, pad);
  if (D > 4096 && D <= 6144)
    return launch_pdl(rmsnorm_rows_reg_kernel<T, OUT_F16, 48>, row_grid(M, 4), dim3(128), 0, s,
                      x, g, u, M, D, pad);
  return launch_pdl(rmsnorm_rows_kernel<T, OUT_F16>, row_grid(M, 8), dim3(256), 0, s, x, g, u, M,
                    D, pad);
}

template <typename T>
cudaError_t launch_post_typed(cudaStream_t s, const float* a, const T* x, const __nv_bfloat16* g,
                              float* y, int M, int D, const PadRows& pad) {
  const int inplace = static_cast<const void*>(x) == static_cast<const void*>(y) ? 1 : 0;
  if (D > 2048 && D <= 4096)
    return launch_pdl(postnorm_residual_reg_kernel<T, 32>, row_grid(M, 4), dim3(128), 0, s, a, x,
                      g, y, M, D, pad, inplace);
  return launch_pdl(postnorm_residual_kernel<T>, row_grid(M, 8), dim3(256), 0, s, a, x, g, y, M,
                    D, pad, inplace);
}

// Padding information is used only when the rows form whole segments.
PadRows checked_pad(const PadRows& pad, int M) {
  if (pad.pad_lens == nullptr || pad.seg_T < 1 || M % pad.seg_T != 0) return PadRows{};
  return pad;
}

}  // namespace

cudaError_t launch_qk_norm_rope(void* Q, long ldq, void* K, long ldk, const void* gamma_q,
                                const void* gamma_k, const int32_t* pos, int M, int H, int H_kv,
                                int d_h, double rope_base, double rope_scale, float query_scale,
                                cudaStream_t stream, const CacheRows& cache) {
  if (M <= 0) return cudaSuccess;
  if (cache.Kc != nullptr && (cache.T < 1 || M % cache.T != 0)) return cudaErrorInvalidValue;
  if (d_h != 128 && d_h != 256) return cudaErrorInvalidValue;
  // Few rows (a decode step): one warp per head-vector step of a row, so the
  // rows' vectors run on many warps at once; else up to kVecUnroll steps per
  // warp.
  const int chunk_u = M <= 64 ? 1 : kVecUnroll;
  const int vpc = (32 / (d_h / 8)) * chunk_u;
  const long items = static_cast<long>(M) * ((H + H_kv + vpc - 1) / vpc);
  const int warps_per_block = 8;
  long blocks = (items + warps_per_block - 1) / warps_per_block;
  const long cap = static_cast<long>(num_sms()) * 4;
  if (blocks > cap) blocks = cap;
  const RopeFreqs freqs = make_rope_freqs(d_h, rope_base, rope_scale);
  // the span-scan CTAs of a local layer's cache (see the kernel)
  int prep = 0;
  if (cache.span_part != nullptr && cache.window > 0) {
    if (cache.Kc == nullptr || cache.T < 1 || cache.nchunk < 1) return cudaErrorInvalidValue;
    prep = cache.nchunk * (M / cache.T);
  }
  auto q = static_cast<__half*>(Q);
  auto k = static_cast<__half*>(K);
  auto gq = static_cast<const __nv_bfloat16*>(gamma_q);
  auto gk = static_cast<const __nv_bfloat16*>(gamma_k);
  const int qk_blocks = static_cast<int>(blocks);
  if (d_h == 256)
    return launch_pdl(qk_norm_rope_kernel<256>, dim3(qk_blocks + prep), dim3(256), 0, stream, q,
                      ldq, k, ldk, gq, gk, pos, M, H, H_kv, freqs, query_scale, cache, chunk_u,
                      qk_blocks);
  if (d_h == 128)
    return launch_pdl(qk_norm_rope_kernel<128>, dim3(qk_blocks + prep), dim3(256), 0, stream, q,
                      ldq, k, ldk, gq, gk, pos, M, H, H_kv, freqs, query_scale, cache, chunk_u,
                      qk_blocks);
  return cudaErrorInvalidValue;
}

cudaError_t launch_rmsnorm_rows(const void* x, int x_dtype, const void* gamma, void* u,
                                int u_dtype, int M, int D, cudaStream_t stream,
                                const PadRows& pad_in) {
  if (M <= 0) return cudaSuccess;
  const PadRows pad = checked_pad(pad_in, M);
  auto g = static_cast<const __nv_bfloat16*>(gamma);
  auto uo = static_cast<uint16_t*>(u);
  if (u_dtype != kBF16 && u_dtype != kF16) return cudaErrorInvalidValue;
  const bool f16 = u_dtype == kF16;
  if (x_dtype == kF32) {
    auto xp = static_cast<const float*>(x);
    return f16 ? launch_rms_typed<float, true>(stream, xp, g, uo, M, D, pad)
               : launch_rms_typed<float, false>(stream, xp, g, uo, M, D, pad);
  }
  if (x_dtype == kBF16) {
    auto xp = static_cast<const __nv_bfloat16*>(x);
    return f16 ? launch_rms_typed<__nv_bfloat16, true>(stream, xp, g, uo, M, D, pad)
               : launch_rms_typed<__nv_bfloat16, false>(stream, xp, g, uo, M, D, pad);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_cast_bf16_f16(const void* src, void* dst, size_t n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  if (n % 8 != 0) return cudaErrorInvalidValue;
  const size_t n8 = n / 8;
  long blocks = static_cast<long>((n8 + 255) / 256);
  const long cap = static_cast<long>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(cast_bf16_f16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                    static_cast<const uint4*>(src), static_cast<uint4*>(dst), n8);
}

namespace {

// One warp per row, 8 columns (one 16-byte load) per lane per step.  A token
// outside [0, V) gives a zero row and records kDevErrBadToken.
__global__ void __launch_bounds__(256) embed_rows_kernel(const int32_t* __restrict__ tokens,
                                                         const __nv_bfloat16* __restrict__ E,
                                                         int V, int D, int M, float scale,
                                                         float* __restrict__ x, int* status) {
  pdl_enter();
  const int m = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (m >= M) return;
  const int t = tokens[m];
  const bool ok = t >= 0 && t < V;
  if (!ok && lane == 0) record_error(status, kDevErrBadToken);
  const __nv_bfloat16* src = E + static_cast<size_t>(ok ? t : 0) * D;
  float* dst = x + static_cast<size_t>(m) * D;
  for (int c = lane * 8; c < D; c += 256) {
    float f[8];
    if (ok) {
      const uint4 r = __ldg(reinterpret_cast<const uint4*>(src + c));
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 v = __bfloat1622float2(h[i]);
        f[2 * i] = v.x * scale;
        f[2 * i + 1] = v.y * scale;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = 0.f;
    }
    reinterpret_cast<float4*>(dst + c)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(dst + c)[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
}

}  // namespace

cudaError_t launch_embed_rows(const int32_t* tokens, const void* E, int V, int D, int M,
                              float scale, float* x, cudaStream_t stream, int* status) {
  if (M <= 0) return cudaSuccess;
  return launch_pdl(embed_rows_kernel, dim3((M + 7) / 8), dim3(256), 0, stream, tokens,
                    static_cast<const __nv_bfloat16*>(E), V, D, M, scale, x, status);
}

cudaError_t launch_postnorm_residual(const float* a, const void* x, int x_dtype,
                                     const void* gamma, float* y, int M, int D,
                                     cudaStream_t stream, const PadRows& pad_in) {
  if (M <= 0) return cudaSuccess;
  const PadRows pad = checked_pad(pad_in, M);
  auto g = static_cast<const __nv_bfloat16*>(gamma);
  if (x_dtype == kF32)
    return launch_post_typed<float>(stream, a, static_cast<const float*>(x), g, y, M, D, pad);
  if (x_dtype == kBF16)
    return launch_post_typed<__nv_bfloat16>(stream, a, static_cast<const __nv_bfloat16*>(x), g, y,
                                            M, D, pad);
  return cudaErrorInvalidValue;
}

}  // namespace g3
