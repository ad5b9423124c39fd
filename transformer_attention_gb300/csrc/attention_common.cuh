// Pieces shared by the two flash-attention kernels ("Gemma 3 Attention
// Block", How it works: Scores): attention.cu (d_h = 256, one query tile per
// work item) and attention_pair.cu (d_h = 128, two query tiles per item).
//
// Work order.  Items are ordered by groups of `gsz` (b, kv head) pairs whose
// K/V fit in L2 together; within a group the heaviest items (latest query
// tokens, for causal layers) come first, the group's (b, j) pairs varying
// fastest.  With a scheduler counter a free CTA takes the next position of
// that order; without one the CTAs walk it in boustrophedon rounds.
#pragma once

#include "ptx.cuh"

namespace g3 {
namespace attn {

constexpr int KV_TILE = 128;   // keys per KV tile

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// One work item: `span` consecutive query tokens t0 .. t0 + span - 1 (times
// the G heads of kv head j) of batch row b, and the KV tiles it visits.
struct Item {
  int b, j, t0, valid, t_last, tile_lo, n_tiles;
  int s_base;   // first key of the first KV tile; tile i starts at s_base + i * KV_TILE
  int last_n;   // keys of the last tile that any row can see, rounded up to 16
  bool pad;     // every token past the valid length: the item only writes zeros
};

// Position p of the heavy-first order -> item.  n_q items of `span` tokens
// cover each (b, j) pair; KV tiles outside the causal band and the window
// (keep t - W < s <= t) are not visited.  By default the KV tiles sit on
// multiples of KV_TILE.  With `from_window` they start at the item's first
// visible key instead, t0 - W + 1 (0 on a global layer), so the item's keys
// t0 - W + 1 .. t_last span ceil((W + span - 1) / KV_TILE) tiles whatever t0
// is, and only the last tile's first last_n keys are visible to any row
// (its S and PV products can stop there).
__device__ __forceinline__ Item decode_item(int p, int span, int n_q, int gsz, int B, int H_kv,
                                            int T, int window, const int32_t* pad_lens,
                                            bool from_window = false) {
  Item it;
  const int BH = B * H_kv;
  const int group = p / (gsz * n_q);
  const int base = group * gsz;
  const int gs = min(gsz, BH - base);
  const int within = p - group * gsz * n_q;
  const int qi = within / gs;
  const int bj = base + within % gs;
  it.b = bj / H_kv;
  it.j = bj % H_kv;
  it.t0 = (n_q - 1 - qi) * span;
  it.valid = T - (pad_lens != nullptr ? pad_lens[it.b] : 0);
  it.pad = it.t0 >= it.valid;
  it.t_last = min(it.t0 + span, it.valid) - 1;
  const int s_lo = window > 0 ? max(0, it.t0 - window + 1) : 0;
  it.tile_lo = s_lo / KV_TILE;
  if (from_window) {
    const int n_keys = it.t_last - s_lo + 1;
    it.s_base = s_lo;
    it.n_tiles = it.pad ? 0 : (n_keys + KV_TILE - 1) / KV_TILE;
    it.last_n = it.pad ? 0 : (n_keys - (it.n_tiles - 1) * KV_TILE + 15) & ~15;
  } else {
    it.s_base = it.tile_lo * KV_TILE;
    it.n_tiles = it.pad ? 0 : it.t_last / KV_TILE - it.tile_lo + 1;
    it.last_n = KV_TILE;
  }
  return it;
}

// Static order: in round r the CTAs take the next gridDim.x positions, in
// reverse on odd rounds, so heavy-first costs even out across CTAs.
__device__ __forceinline__ int static_position(int r) {
  return r * static_cast<int>(gridDim.x) +
         ((r & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                  : static_cast<int>(blockIdx.x));
}

// Dynamic order: the K producer takes positions from the counter `sched`
// (zeroed before each launch) and hands them to the other roles through
// this ring in shared memory; round rr uses slot rr % SLOTS, released by
// CONSUMERS arrivals.  Every wait is bounded; a failed wait returns
// num_items, which ends the caller's loop.
template <int SLOTS, int CONSUMERS>
struct SchedRing {
  uint64_t full[SLOTS], empty[SLOTS];
  int pos[SLOTS];

  __device__ __forceinline__ void init() {
    for (int s = 0; s < SLOTS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), CONSUMERS);
    }
  }
  // The producing thread: position of round rr, published to the ring.
  __device__ __forceinline__ int fetch(int rr, unsigned int* sched, int num_items,
                                       volatile int* abort_flag, int* status, int site) {
    if (sched == nullptr) return static_position(rr);
    const int slot = rr % SLOTS;
    if (rr >= SLOTS && !mbar_wait(smem_u32(&empty[slot]), ((rr / SLOTS) - 1) & 1, abort_flag,
                                  status, site))
      return num_items;
    const int p = static_cast<int>(min(atomicAdd(sched, 1u), static_cast<unsigned>(num_items)));
    *reinterpret_cast<volatile int*>(&pos[slot]) = p;
    mbar_arrive(smem_u32(&full[slot]));
    return p;
  }
  // Any other role (every lane of a warp may call it): position of round rr.
  __device__ __forceinline__ int take(int rr, const unsigned int* sched, int num_items,
                                      volatile int* abort_flag, int* status, int site) {
    if (sched == nullptr) return static_position(rr);
    const int slot = rr % SLOTS;
    if (!mbar_wait(smem_u32(&full[slot]), (rr / SLOTS) & 1, abort_flag, status, site))
      return num_items;
    return *reinterpret_cast<volatile int*>(&pos[slot]);
  }
  // One arrival per consumer (one thread of each consuming warp).
  __device__ __forceinline__ void release(int rr, const unsigned int* sched) {
    if (sched != nullptr) mbar_arrive(smem_u32(&empty[rr % SLOTS]));
  }
};

// (b, kv head) pairs per ordering group.  Global layers: as many as keep
// their K/V (T x d_h x 2 tensors x 2 B) within ~48 MB of L2.  Local layers
// read only a window of K/V per item, shared by the ~W / span consecutive
// query items of the same pair: the group is small enough that the `ctas`
// items in flight hold that many consecutive items of each of its pairs, so
// each K/V tile is read from DRAM about once.  (One group over all 64 pairs
// of the 12B shape spread the items in flight over every pair, and each K/V
// tile was evicted between its reuses: 3.4x the algorithmic DRAM reads.)
inline int l2_group_size(int B, int H_kv, int T, int d_h, int window, int span, int ctas) {
  const double kv_bytes = static_cast<double>(T) * d_h * 2.0 * 2.0;
  int gsz = window > 0 ? ctas / ((window + span - 1) / span + 1)
                       : static_cast<int>(48.0 * 1024 * 1024 / kv_bytes);
  return gsz < 1 ? 1 : (gsz > B * H_kv ? B * H_kv : gsz);
}

}  // namespace attn
}  // namespace g3
