// The visible span of a local layer's cache, shared by the cache-attention
// launcher (decode.cu) and the decode-step prologue (elementwise.cu), which
// computes it in the same launch as the QK-norm/RoPE of the new tokens.
//
// Slot s of batch row b can be visible to a valid query of the row only if
// its stored position p_s >= 0 and p_s > min_t(pos_t) - W ("Gemma 3
// Attention Block", How it works: Cache keeps the positions for the sliding
// mask).  The slots [end, end + T) hold the new tokens, whose positions are
// taken from the query positions (pad tokens are empty), so the scan never
// reads slots that the same launch writes.
#pragma once

#include <climits>
#include <cstdint>

namespace g3 {

constexpr int kSpanChunk = 4096;   // slots per CTA of the scan (256 threads x 16)

__device__ __forceinline__ int span_warp_min(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One CTA of 256 threads: the first slot of chunk c (slots [c * kSpanChunk,
// (c + 1) * kSpanChunk) within [0, end + T)) that a valid query of row b can
// see, or INT_MAX, written to span_part[b * nchunk + c].
__device__ __forceinline__ void kv_span_chunk(const int32_t* __restrict__ posc,
                                              const int32_t* __restrict__ qpos,
                                              const int32_t* __restrict__ pad_lens, int T, int S,
                                              int end, int window, int nchunk,
                                              int32_t* __restrict__ span_part, int c, int b) {
  __shared__ int red[8];
  const int valid = T - (pad_lens != nullptr ? pad_lens[b] : 0);
  int qmin = INT_MAX;
  for (int t = threadIdx.x; t < valid; t += blockDim.x)
    qmin = min(qmin, qpos[static_cast<size_t>(b) * T + t]);
  qmin = span_warp_min(qmin);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = qmin;
  __syncthreads();
  qmin = INT_MAX;
  for (int i = 0; i < 8; ++i) qmin = min(qmin, red[i]);
  __syncthreads();
  const long long thr = static_cast<long long>(qmin) - window;
  // Each thread owns 16 consecutive slots of the chunk; stored slots are read
  // at once (four 16-byte loads when the row is 16-byte aligned), so the scan
  // costs one memory round trip.
  const int s_end = min(end + T, (c + 1) * kSpanChunk);
  const int s0 = c * kSpanChunk + static_cast<int>(threadIdx.x) * 16;
  const int32_t* row = posc + static_cast<size_t>(b) * S;
  int v[16];
  if ((reinterpret_cast<uintptr_t>(row + s0) & 15u) == 0 && s0 + 16 <= min(s_end, end)) {
    const int4* q = reinterpret_cast<const int4*>(row + s0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int4 x = __ldg(q + i);
      v[4 * i] = x.x;
      v[4 * i + 1] = x.y;
      v[4 * i + 2] = x.z;
      v[4 * i + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int s = s0 + i;
      const int t = s - end;   // new token t (0 <= t < T) in slot end + t
      v[i] = s >= s_end ? -1
             : s < end  ? __ldg(row + s)
             : (t < valid ? qpos[static_cast<size_t>(b) * T + t] : -1);
    }
  }
  int best = INT_MAX;
#pragma unroll
  for (int i = 15; i >= 0; --i)
    if (v[i] >= 0 && static_cast<long long>(v[i]) > thr) best = s0 + i;
  best = span_warp_min(best);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    int m = INT_MAX;
    for (int i = 0; i < 8; ++i) m = min(m, red[i]);
    span_part[static_cast<size_t>(b) * nchunk + c] = m;
  }
}

}  // namespace g3
