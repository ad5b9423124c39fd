// KV-cache path of the attention layer ("Gemma 3 Attention Block", How it
// works: Cache): the write of the new tokens' K', V and positions into a
// left-aligned cache, and attention of those tokens over the cache's slots.
//
// Mask over slots (one batch row, query token t written to slot end + t):
//   slot s is visible  <=>  s <= end + t, its stored position p_s >= 0 (an
//   empty slot stores -1), and on a local layer pos_t - W < p_s < pos_t + W
//   (the sliding mask of the same section evaluated on the stored positions).
//
// Attention over a cache is bound by HBM: every visible slot's K' and V
// (2 x d_h fp16) are read once and used by only G x T query rows, which is far
// too few rows for a tensor-core tile.  The kernel therefore streams K'/V
// tiles of 32 slots through a TMA ring in shared memory and does the two small
// contractions on the CUDA cores in fp32.  The visible slot range of a batch
// row is split across CTAs (two resident per SM); each CTA keeps an online
// softmax per query row and writes an unnormalised partial (m, l, o) that a
// second kernel merges.  On a local layer the first slot any query of the row
// can see is found first (by the decode-step prologue kernel in its own
// launch, or else by a small kernel here), so CTAs cover only the window.
#include <algorithm>
#include <climits>
#include <cmath>

#include "decode_span.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace g3 {

namespace {

constexpr int kSlots = 32;         // slots per tile: one per lane in the logits phase
constexpr int kCWarps = 4;         // consumer warps; warp 4 issues the TMA loads
constexpr int kDecThreads = (kCWarps + 1) * 32;
constexpr int kMaxSplitCtas = 2048;
constexpr int kMaxCombineSplits = 256;   // splits per row the combine kernel holds weights for
constexpr int kMinSplitTiles = 2;        // fewest tiles worth a split of its own
constexpr float kLog2e = 1.4426950408889634f;

enum { kSiteDecFull = 40, kSiteDecEmpty = 41, kSiteDecIssued = 42 };

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Bounded wait (whole warp) until the producer has issued tile i; false on
// timeout or when the CTA was aborted.
__device__ __forceinline__ bool wait_issued(int* issued, int i, volatile int* abort_flag,
                                            int* status) {
  const volatile int* v = issued;
  bool ok = true;
  if (*v <= i) {
    const uint64_t t0 = globaltimer();
    while (*v <= i) {
      if (*abort_flag) {
        ok = false;
        break;
      }
      if (globaltimer() - t0 > kWaitTimeoutNs) {
        record_error(status, kDevErrTimeoutBase + kSiteDecIssued);
        *abort_flag = 1;
        ok = false;
        break;
      }
    }
  }
  __threadfence_block();
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void unpack8(const uint4& r, float (&f)[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __half22float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}
__device__ __forceinline__ void unpack4(const uint2& r, float (&f)[4]) {
  const __half2* h = reinterpret_cast<const __half2*>(&r);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float2 v = __half22float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

// ---------------------------------------------------------------- cache write
// One CTA per new token (t, b): copies its K' and V rows (KVD = H_kv * d_h
// fp16 each) into slot end + t and stores its position (-1 for a pad token).
__global__ void __launch_bounds__(128) kv_cache_append_kernel(
    const __half* __restrict__ K_rows, const __half* __restrict__ V_rows, long ld,
    const int32_t* __restrict__ segment_pos, const int32_t* __restrict__ pad_lens, int T, int S,
    int end, int KVD, __half* __restrict__ Kc, __half* __restrict__ Vc,
    int32_t* __restrict__ posc) {
  pdl_enter();
  const int t = blockIdx.x, b = blockIdx.y;
  const size_t src = (static_cast<size_t>(b) * T + t) * ld;
  const size_t slot = static_cast<size_t>(b) * S + end + t;
  const uint4* ks = reinterpret_cast<const uint4*>(K_rows + src);
  const uint4* vs = reinterpret_cast<const uint4*>(V_rows + src);
  uint4* kd = reinterpret_cast<uint4*>(Kc + slot * KVD);
  uint4* vd = reinterpret_cast<uint4*>(Vc + slot * KVD);
  for (int i = threadIdx.x; i < KVD / 8; i += blockDim.x) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
  if (threadIdx.x == 0) {
    const int valid = T - (pad_lens != nullptr ? pad_lens[b] : 0);
    posc[slot] = t < valid ? segment_pos[static_cast<size_t>(b) * T + t] : -1;
  }
}

// ---------------------------------------------------------------- span
// Local layers: CTA (c, b) writes the first slot of chunk c that a valid
// query of row b can see, or INT_MAX (decode_span.cuh).
__global__ void __launch_bounds__(256) kv_span_kernel(
    const int32_t* __restrict__ posc, const int32_t* __restrict__ qpos,
    const int32_t* __restrict__ pad_lens, int T, int S, int end, int window, int nchunk,
    int32_t* __restrict__ span_part) {
  pdl_enter();
  kv_span_chunk(posc, qpos, pad_lens, T, S, end, window, nchunk, span_part, blockIdx.x,
                blockIdx.y);
}

// ---------------------------------------------------------------- attention
template <int DH, int RB>
struct DecCfg {
  static constexpr int NCH = DH / 64;                  // 128-byte column chunks of a row
  static constexpr int BOX = kSlots * 128;             // one {64 ch, 32 slots} box, swizzled
  static constexpr int TILE = 2 * NCH * BOX;           // K' and V of one tile
  static constexpr int NST = DH == 256 ? 3 : 6;        // ring stages (96 KB either way)
  static constexpr int RING = NST * TILE;
  static constexpr int QS = RB * DH * 4;               // fp32 query rows
  static constexpr int PS = kCWarps * RB * kSlots * 4; // per-warp probabilities
  static constexpr int REC = DH + 4;                   // merge record: m, l, 2 pad, o[DH]
  static constexpr int MERGE = kCWarps * RB * REC * 4; // reuses the ring after the last tile
  static constexpr int SMEM = 1024 + RING + QS + PS;
  static constexpr int VPL = DH / 32;                  // V channels per lane
  static_assert(MERGE <= RING, "merge records must fit in the ring");
  static_assert(SMEM <= 112 * 1024, "two CTAs per SM");
};

struct DecParams {
  const __half* Q;            // [B, T, H, DH] (query scale applied)
  const int32_t* posc;        // [B, S] stored positions
  const int32_t* qpos;        // [B, T] query positions
  const int32_t* pad_lens;    // [B] or null
  const int32_t* span_part;   // [B, nchunk] (local layers) or null
  float* part;                // [B*T*H, nsplit, REC] when nsplit > 1
  void* O;                    // [B, T, H, DH] when nsplit == 1
  int o_f16, B, T, S, H, H_kv, end, window, nsplit, nchunk, tq, ntg;
  int* status;
};

template <int DH, int RB>
__global__ void __launch_bounds__(kDecThreads, 2)
    decode_attn_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const DecParams p) {
  pdl_enter();
  using C = DecCfg<DH, RB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  float* qs = reinterpret_cast<float*>(smem + C::RING);            // [RB][DH]
  float* ps = reinterpret_cast<float*>(smem + C::RING + C::QS);    // [kCWarps][RB][kSlots]
  __shared__ __align__(8) uint64_t full[C::NST], empty[C::NST];
  __shared__ int abort_flag;
  // Tiles whose loads the producer has issued.  Tiles go to the consumer
  // warps round-robin and to the stages modulo NST, so a warp can come back to
  // a stage two or more fills ahead of the barrier's phase, where a parity
  // wait alone is ambiguous; waiting first for `issued > i` guarantees the
  // stage's previous fill has completed, which makes the parity wait exact.
  __shared__ int issued;
  __shared__ int row_lim[RB];          // last visible slot of row r (end + t), -1 = no query
  __shared__ long long row_thr[RB];    // stored position must exceed this ...
  __shared__ long long row_top[RB];    // ... and stay below this
  __shared__ int rng[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, j = blockIdx.y;
  const int b = blockIdx.z / p.ntg, tg = blockIdx.z % p.ntg;
  const int G = p.H / p.H_kv;
  const int t0 = tg * p.tq;
  const int ntok = min(p.tq, p.T - t0);
  const int R = ntok * G;
  const int valid = p.T - (p.pad_lens != nullptr ? p.pad_lens[b] : 0);

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    abort_flag = 0;
    issued = 0;
    fence_barrier_init();
  }
  if (tid < RB) {
    int lim = -1;
    long long thr = LLONG_MIN, top = LLONG_MAX;
    if (tid < R) {
      const int t = t0 + tid / G;
      if (t < valid) {
        lim = p.end + t;
        if (p.window > 0) {
          const long long qp = p.qpos[static_cast<size_t>(b) * p.T + t];
          thr = qp - p.window;
          top = qp + p.window;
        }
      }
    }
    row_lim[tid] = lim;
    row_thr[tid] = thr;
    row_top[tid] = top;
  }
  if (warp == 1) {
    // Visible slots of this CTA's rows lie in [lo, hi); split them evenly
    // (in whole tiles) over the nsplit CTAs of (b, j, tg).
    int lo = 0;
    if (p.span_part != nullptr) {
      lo = INT_MAX;
      for (int i = lane; i < p.nchunk; i += 32)
        lo = min(lo, p.span_part[static_cast<size_t>(b) * p.nchunk + i]);
      lo = warp_min_i(lo);
    }
    const int t_last = min(t0 + ntok, valid) - 1;
    const int hi = t_last >= t0 ? p.end + t_last + 1 : 0;
    lo = min(lo, hi);
    const int span = hi - lo;
    int chunk = (span + p.nsplit - 1) / p.nsplit;
    chunk = (chunk + kSlots - 1) / kSlots * kSlots;
    const long long a = static_cast<long long>(lo) + static_cast<long long>(split) * chunk;
    const int e = static_cast<int>(min(static_cast<long long>(hi), a + chunk));
    const int s = static_cast<int>(min(a, static_cast<long long>(e)));
    if (lane == 0) {
      rng[0] = s;
      rng[1] = e;
    }
  }
  // Query rows in shared memory as fp32, pre-multiplied by log2(e) so the
  // softmax runs on exp2.
  for (int i = tid; i < RB * DH / 8; i += kDecThreads) {
    const int r = (i * 8) / DH, c = (i * 8) % DH;
    float f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = 0.f;
    if (r < R) {
      const int t = t0 + r / G, h = j * G + r % G;
      unpack8(__ldg(reinterpret_cast<const uint4*>(
                  p.Q + ((static_cast<size_t>(b) * p.T + t) * p.H + h) * DH + c)),
              f);
    }
    float4* dst = reinterpret_cast<float4*>(qs + r * DH + c);
    dst[0] = make_float4(f[0] * kLog2e, f[1] * kLog2e, f[2] * kLog2e, f[3] * kLog2e);
    dst[1] = make_float4(f[4] * kLog2e, f[5] * kLog2e, f[6] * kLog2e, f[7] * kLog2e);
  }
  __syncthreads();
  const int s_lo = rng[0], s_hi = rng[1];
  const int n_tiles = (s_hi - s_lo + kSlots - 1) / kSlots;

  if (warp == kCWarps) {
    // ---------------- producer: K'/V tiles of 32 slots into the ring
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % C::NST;
        if (i >= C::NST && !mbar_wait(smem_u32(&empty[st]), ((i / C::NST) - 1) & 1, &abort_flag,
                                      p.status, kSiteDecEmpty))
          break;
        const uint32_t bar = smem_u32(&full[st]);
        mbar_arrive_expect_tx(bar, C::TILE);
        uint8_t* kd = ring + st * C::TILE;
        uint8_t* vd = kd + C::NCH * C::BOX;
        const int s0 = s_lo + i * kSlots;
#pragma unroll
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_4d(smem_u32(kd + c * C::BOX), &tmK, bar, c * 64, j, s0, b);
          tma_load_4d(smem_u32(vd + c * C::BOX), &tmV, bar, c * 64, j, s0, b);
        }
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&issued) = i + 1;
      }
      // Every issued load lands before the CTA may exit.
      const int n_issued = *reinterpret_cast<volatile int*>(&issued);
      for (int i = max(0, n_issued - C::NST); i < n_issued; ++i)
        mbar_wait_drain(smem_u32(&full[i % C::NST]), (i / C::NST) & 1);
    }
    return;
  }

  // ---------------- consumers: warp w takes tiles w, w+4, ...
  float m[RB], l[RB], o[RB][C::VPL];
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int k = 0; k < C::VPL; ++k) o[r][k] = 0.f;
  }
  float* pw = ps + warp * RB * kSlots;

  for (int i = warp; i < n_tiles; i += kCWarps) {
    const int st = i % C::NST;
    const int s = s_lo + i * kSlots + lane;
    const int pos_s = s < s_hi ? __ldg(&p.posc[static_cast<size_t>(b) * p.S + s]) : -1;
    if (!wait_issued(&issued, i, &abort_flag, p.status)) break;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&full[st]), (i / C::NST) & 1,
                                                      &abort_flag, p.status, kSiteDecFull));
    if (!ok) break;
    const uint8_t* kt = ring + st * C::TILE;
    const uint8_t* vt = kt + C::NCH * C::BOX;

    // logits: lane = slot, all DH channels of its K' row against every query row
    float acc[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) acc[r] = 0.f;
#pragma unroll 4
    for (int u = 0; u < DH / 8; ++u) {
      const int c = u >> 3, uu = u & 7;
      const uint4 kr =
          *reinterpret_cast<const uint4*>(kt + c * C::BOX + lane * 128 + ((uu ^ (lane & 7)) << 4));
      float kf[8];
      unpack8(kr, kf);
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        if (r < R) {
          const float4 qa = *reinterpret_cast<const float4*>(qs + r * DH + u * 8);
          const float4 qb = *reinterpret_cast<const float4*>(qs + r * DH + u * 8 + 4);
          float a = acc[r];
          a = fmaf(qa.x, kf[0], a);
          a = fmaf(qa.y, kf[1], a);
          a = fmaf(qa.z, kf[2], a);
          a = fmaf(qa.w, kf[3], a);
          a = fmaf(qb.x, kf[4], a);
          a = fmaf(qb.y, kf[5], a);
          a = fmaf(qb.z, kf[6], a);
          a = fmaf(qb.w, kf[7], a);
          acc[r] = a;
        }
      }
    }

    // mask and online softmax (log2 domain)
    float scale[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      scale[r] = 1.f;
      if (r < R) {
        const long long ps64 = pos_s;
        const bool vis = pos_s >= 0 && s <= row_lim[r] && ps64 > row_thr[r] && ps64 < row_top[r];
        const float x = vis ? acc[r] : -INFINITY;
        const float mn = fmaxf(m[r], warp_max(x));
        float pr = 0.f;
        if (mn != -INFINITY) {
          scale[r] = ex2_approx(m[r] - mn);
          pr = ex2_approx(x - mn);
        }
        l[r] = l[r] * scale[r] + pr;
        m[r] = mn;
        pw[r * kSlots + lane] = pr;
      }
    }
    __syncwarp();

    // V mix: lane owns VPL channels, loops over the tile's slots
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
      for (int k = 0; k < C::VPL; ++k) o[r][k] *= scale[r];
#pragma unroll 2
    for (int sl = 0; sl < kSlots; sl += 4) {
      float4 p4[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r)
        p4[r] = r < R ? *reinterpret_cast<const float4*>(pw + r * kSlots + sl)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int row = sl + q;
        float vf[C::VPL];
        if constexpr (DH == 256) {
          const uint4 vr = *reinterpret_cast<const uint4*>(
              vt + (lane >> 3) * C::BOX + row * 128 + (((lane & 7) ^ (row & 7)) << 4));
          unpack8(vr, vf);
        } else {
          const uint2 vr = *reinterpret_cast<const uint2*>(
              vt + (lane >> 4) * C::BOX + row * 128 + ((((lane & 15) >> 1) ^ (row & 7)) << 4) +
              ((lane & 1) << 3));
          unpack4(vr, vf);
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          if (r < R) {
            const float pv = q == 0 ? p4[r].x : q == 1 ? p4[r].y : q == 2 ? p4[r].z : p4[r].w;
#pragma unroll
            for (int k = 0; k < C::VPL; ++k) o[r][k] = fmaf(pv, vf[k], o[r][k]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
  }

#pragma unroll
  for (int r = 0; r < RB; ++r) l[r] = warp_sum(l[r]);

  // Merge the four warps (records in the ring: every tile has been consumed,
  // so no copy is still writing there).
  named_barrier(1, kCWarps * 32);
  float* mg = reinterpret_cast<float*>(ring);
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    if (r < R) {
      float* rec = mg + (warp * RB + r) * C::REC;
      if (lane == 0) {
        rec[0] = m[r];
        rec[1] = l[r];
      }
#pragma unroll
      for (int k = 0; k < C::VPL; ++k) rec[4 + lane * C::VPL + k] = o[r][k];
    }
  }
  named_barrier(1, kCWarps * 32);
  for (int idx = tid; idx < R * DH; idx += kCWarps * 32) {
    const int r = idx / DH, c = idx % DH;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCWarps; ++w) M = fmaxf(M, mg[(w * RB + r) * C::REC]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kCWarps; ++w) {
        const float* rec = mg + (w * RB + r) * C::REC;
        const float f = ex2_approx(rec[0] - M);
        L += f * rec[1];
        acc += f * rec[4 + c];
      }
    }
    const int t = t0 + r / G, h = j * G + r % G;
    const size_t orow = (static_cast<size_t>(b) * p.T + t) * p.H + h;
    if (p.nsplit == 1) {
      const float v = L > 0.f ? acc / L : 0.f;
      if (p.o_f16)
        static_cast<__half*>(p.O)[orow * DH + c] = __float2half_rn(v);
      else
        static_cast<__nv_bfloat16*>(p.O)[orow * DH + c] = __float2bfloat16_rn(v);
    } else {
      float* rec = p.part + (orow * p.nsplit + split) * C::REC;
      if (c == 0) {
        rec[0] = M;
        rec[1] = L;
      }
      rec[4 + c] = acc;
    }
  }
}

// ---------------------------------------------------------------- combine
// One warp per (b, t, h) row: O = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i.
// One CTA of DH threads per (b, t, h) row; thread c owns channel c.
template <int DH>
__global__ void __launch_bounds__(DH) decode_combine_kernel(const float* __restrict__ part,
                                                            void* O, int o_f16, int nsplit) {
  pdl_enter();
  constexpr int REC = DH + 4, NW = DH / 32;
  __shared__ float fw[NW][kMaxCombineSplits];
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31, c = threadIdx.x;
  const size_t row = blockIdx.x;
  const float* base = part + row * nsplit * REC;
  // weights 2^(m_i - M) and their l-weighted total, lanes over splits (each
  // warp computes its own copy; the records are L2-resident)
  float M = -INFINITY;
  for (int i = lane; i < nsplit; i += 32) M = fmaxf(M, base[static_cast<size_t>(i) * REC]);
  M = warp_max(M);
  float L = 0.f;
  for (int i = lane; i < nsplit; i += 32) {
    const float* rec = base + static_cast<size_t>(i) * REC;
    const float f = M == -INFINITY ? 0.f : ex2_approx(rec[0] - M);
    fw[wid][i] = f;
    L += f * rec[1];
  }
  L = warp_sum(L);
  __syncwarp();
  float acc = 0.f;
#pragma unroll 8
  for (int i = 0; i < nsplit; ++i)
    acc = fmaf(fw[wid][i], __ldg(base + static_cast<size_t>(i) * REC + 4 + c), acc);
  const float v = L > 0.f ? acc / L : 0.f;
  if (o_f16)
    static_cast<__half*>(O)[row * DH + c] = __float2half_rn(v);
  else
    static_cast<__nv_bfloat16*>(O)[row * DH + c] = __float2bfloat16_rn(v);
}

// ---------------------------------------------------------------- planning
struct DecPlan {
  int rb, tq, ntg, units;
};

DecPlan plan_rows(int B, int T, int H, int H_kv) {
  const int G = H / H_kv;
  const int want = T * G < 8 ? T * G : 8;
  int rb = want <= 2 ? 2 : (want <= 4 ? 4 : 8);
  if (rb < G) rb = G;
  DecPlan d;
  d.rb = rb;
  d.tq = rb / G;
  d.ntg = (T + d.tq - 1) / d.tq;
  d.units = B * H_kv * d.ntg;
  return d;
}

int max_splits(const DecPlan& d) {
  int m = kMaxSplitCtas / d.units;
  if (m > kMaxCombineSplits) m = kMaxCombineSplits;
  return m < 1 ? 1 : m;
}

template <int DH, int RB>
cudaError_t launch_decode_cfg(const CUtensorMap& tk, const CUtensorMap& tv, const DecParams& p,
                              dim3 grid, cudaStream_t stream) {
  using C = DecCfg<DH, RB>;
  auto kern = decode_attn_kernel<DH, RB>;
  if (cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::SMEM)) return e;
  return launch_pdl(kern, grid, dim3(kDecThreads), C::SMEM, stream, tk, tv, p);
}

}  // namespace

cudaError_t launch_kv_cache_append(const void* K_rows, const void* V_rows, long ld,
                                   const int32_t* segment_pos, const int32_t* pad_lens, int B,
                                   int T, int S, int end, int KVD, void* K_cache, void* V_cache,
                                   int32_t* pos_cache, cudaStream_t stream) {
  if (B <= 0 || T <= 0) return cudaSuccess;
  if (B > 65535) return cudaErrorInvalidValue;
  return launch_pdl(kv_cache_append_kernel, dim3(T, B), dim3(128), 0, stream,
                    static_cast<const __half*>(K_rows), static_cast<const __half*>(V_rows), ld,
                    segment_pos, pad_lens, T, S, end, KVD, static_cast<__half*>(K_cache),
                    static_cast<__half*>(V_cache), pos_cache);
}

CachedAttnLayout cached_attention_layout(void* ws, int B, int T, int S, int H, int H_kv, int d_h) {
  const DecPlan d = plan_rows(B, T, H, H_kv);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  CachedAttnLayout L;
  L.nchunk = (S + kSpanChunk - 1) / kSpanChunk;
  const size_t span = up(static_cast<size_t>(B) * L.nchunk * 4);
  const size_t part = up(static_cast<size_t>(B) * T * H * max_splits(d) * (d_h + 4) * 4);
  uint8_t* w = static_cast<uint8_t*>(ws);
  L.span_part = reinterpret_cast<int32_t*>(w);
  L.part = reinterpret_cast<float*>(w + span);
  L.bytes = span + part;
  return L;
}

size_t cached_attention_ws_bytes(int B, int T, int S, int H, int H_kv, int d_h) {
  return cached_attention_layout(nullptr, B, T, S, H, H_kv, d_h).bytes;
}

int cached_span_chunks(int T, int end) { return (end + T + kSpanChunk - 1) / kSpanChunk; }

cudaError_t launch_cached_attention(const void* Q, const void* K_cache, const void* V_cache,
                                    const int32_t* pos_cache, const int32_t* qpos,
                                    const int32_t* pad_lens, void* O, int o_dtype, int B, int T,
                                    int S, int end, int H, int H_kv, int d_h, int window,
                                    void* ws, cudaStream_t stream, int* status, bool prepared) {
  if (B <= 0 || T <= 0) return cudaSuccess;
  if (o_dtype != kBF16 && o_dtype != kF16) return cudaErrorInvalidValue;
  const DecPlan d = plan_rows(B, T, H, H_kv);
  if (static_cast<long long>(B) * d.ntg > 65535 || B > 65535 || H_kv > 65535)
    return cudaErrorInvalidValue;
  const int hi = end + T;
  const int nchunk = cached_span_chunks(T, end);
  const CachedAttnLayout lay = cached_attention_layout(ws, B, T, S, H, H_kv, d_h);
  int32_t* span_part = lay.span_part;
  float* part = lay.part;

  // Splits: enough CTAs for two per SM, but at least kMinSplitTiles tiles
  // each over the span the rows are expected to see (a local layer's window
  // plus the new tokens; empty slots or position gaps only make the real span
  // longer, which costs time, never correctness), within the workspace bound.
  int nsplit = (2 * num_sms()) / d.units;
  const long long est = window > 0 ? std::min<long long>(hi, static_cast<long long>(window) + T)
                                   : static_cast<long long>(hi);
  const long long by_span = (est + kMinSplitTiles * kSlots - 1) / (kMinSplitTiles * kSlots);
  if (nsplit > by_span) nsplit = static_cast<int>(by_span);
  if (nsplit > max_splits(d)) nsplit = max_splits(d);
  if (nsplit < 1) nsplit = 1;

  // The span scan of a local layer, unless the decode-step prologue already
  // wrote it (`prepared`).
  if (window > 0 && !prepared) {
    cudaError_t e = launch_pdl(kv_span_kernel, dim3(nchunk, B), dim3(256), 0, stream, pos_cache,
                               qpos, pad_lens, T, S, end, window, nchunk, span_part);
    if (e != cudaSuccess) return e;
  }

  // K'/V caches [B, S, H_kv, d_h]: box {64 channels, 1 head, 32 slots, 1 row}.
  CUtensorMap tk, tv;
  const uint64_t dims[4] = {static_cast<uint64_t>(d_h), static_cast<uint64_t>(H_kv),
                            static_cast<uint64_t>(S), static_cast<uint64_t>(B)};
  const uint64_t str[3] = {static_cast<uint64_t>(d_h) * 2, static_cast<uint64_t>(H_kv) * d_h * 2,
                           static_cast<uint64_t>(S) * H_kv * d_h * 2};
  const uint32_t box[4] = {64, 1, kSlots, 1};
  if (!encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, K_cache, dims, str, box) ||
      !encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, V_cache, dims, str, box))
    return cudaErrorInvalidValue;

  DecParams p;
  p.Q = static_cast<const __half*>(Q);
  p.posc = pos_cache;
  p.qpos = qpos;
  p.pad_lens = pad_lens;
  p.span_part = window > 0 ? span_part : nullptr;
  p.part = part;
  p.O = O;
  p.o_f16 = o_dtype == kF16 ? 1 : 0;
  p.B = B;
  p.T = T;
  p.S = S;
  p.H = H;
  p.H_kv = H_kv;
  p.end = end;
  p.window = window > 0 ? window : 0;
  p.nsplit = nsplit;
  p.nchunk = nchunk;
  p.tq = d.tq;
  p.ntg = d.ntg;
  p.status = status;
  const dim3 grid(nsplit, H_kv, B * d.ntg);
  cudaError_t e = cudaErrorInvalidValue;
#define G3_DEC_CASE(DH_, RB_) \
  if (d_h == DH_ && d.rb == RB_) e = launch_decode_cfg<DH_, RB_>(tk, tv, p, grid, stream);
  G3_DEC_CASE(256, 2)
  G3_DEC_CASE(256, 4)
  G3_DEC_CASE(256, 8)
  G3_DEC_CASE(128, 2)
  G3_DEC_CASE(128, 4)
  G3_DEC_CASE(128, 8)
#undef G3_DEC_CASE
  if (e != cudaSuccess || nsplit == 1) return e;
  const int rows = B * T * H;
  if (d_h == 256)
    return launch_pdl(decode_combine_kernel<256>, dim3(rows), dim3(256), 0, stream,
                      static_cast<const float*>(part), O, p.o_f16, nsplit);
  return launch_pdl(decode_combine_kernel<128>, dim3(rows), dim3(128), 0, stream,
                    static_cast<const float*>(part), O, p.o_f16, nsplit);
}

}  // namespace g3
