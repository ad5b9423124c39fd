// Flash-style attention forward on tcgen05 tensor cores.
//
// Computes, per query row t of batch row b and query head h (kv head
// j = h / G, "Gemma 3 Attention Block", How it works: Scores and the GQA
// reshape):
//   logits[s] = sum_c Q'[b,t,h,c] K'[b,s,j,c]          (query scale already in Q')
//   keep s iff s <= t, s < valid_b and (global or s > t - W)   (causal+padding
//        mask times the sliding mask; blocked logits contribute exp(.) = 0)
//   O[b,t,h,:] = softmax_s(logits) @ V[b,:,j,:]
// with an fp32 online softmax; O is stored as bf16 or fp16.  Rows
// t >= valid_b are written as zeros.
//
// One CTA owns 128 query rows: TQ = 128/G consecutive tokens x the G query
// heads that share kv head j, so every K/V tile loaded from memory feeds all G
// heads of its group.  KV tiles of 128 keys outside the causal band / window
// are never visited (local layers cost O(T*W)); only tiles that straddle the
// band edge, the window edge or the valid length apply an element mask.  The
// tiles start at the item's first visible key (t0 - W + 1, or 0), so an item
// spans ceil((W + TQ - 1) / 128) tiles, and the last tile's S and PV products
// stop at the keys some row of the item can see.
// Work items are ordered in groups of (b, kv-head) pairs whose K/V fit in L2,
// heaviest query tiles first within a group, and the persistent CTAs (one per
// SM) take the next position from a counter (or walk the order in
// boustrophedon rounds without one), so the items in flight stream the same
// K/V tiles through L2 together and causal costs even out
// (attention_common.cuh).
//
// Warp roles (16 warps, four warpgroups):
//   warp 0      TMA producer of Q (once per item, 4-D box over [B,T,H,d_h])
//               and K_i, released per half of its channels
//   warp 2      TMA producer of V_i, released per half of its keys
//   warp 1      TMEM allocation + MMA issue (the whole warp runs the loop,
//               one elected lane issues every tcgen05 instruction):
//                 S  = Q K_i^T   (SS, M=128 N=128, K=d_h)      -> TMEM S
//                 O += P_i V_i   (TS: P_i read from TMEM,      M=128 N=d_h K=128)
//   warps 4-7   softmax: row r of S lives in TMEM lane r, and thread r holds
//               all 128 columns of it in registers (no exchange between
//               threads); it rescales O when its row max grows and hands the
//               item's row sum to the epilogue.
//   warps 8-15  epilogue, two warpgroups, one per 128-column half of O: at the
//               end of an item they read O from TMEM, release it to the next
//               item's first PV, then normalise and store it while the softmax
//               already works on the next item's tiles.
// Registers move from the producer / MMA warpgroup to the softmax warpgroup
// (setmaxnreg).
// TMEM columns: S buffers at 0-127 and 128-255, O at 256-511.  (d_h = 128
// runs in attention_pair.cu, two query tiles per CTA.)  The softmax writes P
// (fp16 pairs) over the first 64 columns of the S buffer it has just read,
// and PV reads it from there; the S of tile i + NS reuses the buffer, issued
// after PV_i by the same warp,
// so the tensor pipe's in-order execution keeps the two apart and no
// barrier is needed to release S: the next S starts as soon as the tensor
// pipe is free.  On tiles without masked elements the row max comes from the
// TMEM load's own max reduction (tcgen05.ld.red).  O is rescaled in TMEM only
// when a row max grows by more than 2^8.
#include "attention_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace g3 {

namespace {

constexpr int NUM_WARPS = 16;
constexpr int THREADS = NUM_WARPS * 32;
constexpr int BM = 128;   // query rows per CTA
constexpr int BN = attn::KV_TILE;   // keys per KV tile
constexpr int SM_WARPS = 4;    // softmax warps
constexpr int EPI_WARPS = 8;   // epilogue warps
constexpr uint32_t CHUNK = 128 * 128;  // one 128-row x 64-element (128 B) swizzled chunk
constexpr uint32_t O_COL = 256;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units
// Registers per thread: the launch gives every thread 65536 / 512 = 128;
// the producer / MMA warpgroup drops to REGS_LOW, the softmax warpgroup
// rises to REGS_SOFT (a whole 128-column row of S in registers) and the
// epilogue warpgroups take REGS_EPI (a 128-column half row of O, packed).
constexpr int REGS_LAUNCH = 128;
constexpr int REGS_LOW = 72, REGS_SOFT = 200, REGS_EPI = 120;
constexpr int REGS_SPLIT = 128 * (REGS_LOW + REGS_SOFT + 2 * REGS_EPI);
static_assert(REGS_SPLIT <= THREADS * REGS_LAUNCH, "register split above the launch allocation");

enum : int {
  kSiteQ = 11, kSiteKEmpty, kSiteVEmpty, kSiteKFull, kSiteSFree, kSitePFull, kSiteVFull,
  kSiteSFull, kSiteORescale, kSitePFree, kSiteOFinal, kSiteLFull, kSiteSchedFull,
  kSiteSchedEmpty
};

// Dynamic order: with a scheduler counter the K producer takes positions of
// the heavy-first order from it (a CTA that is free takes the heaviest item
// left) and hands them to the other roles through a ring in shared memory.
constexpr int SCHED_SLOTS = 4;
constexpr int SCHED_CONSUMERS = 2 + SM_WARPS + EPI_WARPS;   // V producer, MMA, softmax, epilogue

// Columns outside [lo, hi] of a 32-column group (indices relative to the
// group, shifted by its first column) become -inf.
__device__ __forceinline__ void mask32(uint32_t (&r)[32], int first, int hi) {
#pragma unroll
  for (int c = 0; c < 32; ++c)
    if (first + c < 0 || first + c > hi) r[c] = 0xff800000u;   // -inf
}

// exp2(s log2 e - m) of 32 columns (16 pairs): packed fp16 pairs to p[0..15]
// and the sums into acc.
__device__ __forceinline__ void exp_pack16(const uint32_t (&s)[32], uint32_t* p, float2 (&acc)[4],
                                           float2 l2e, float2 negm) {
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float2 xx =
        __ffma2_rn(make_float2(__uint_as_float(s[2 * k]), __uint_as_float(s[2 * k + 1])), l2e,
                   negm);
    const float2 pp = make_float2(attn::ex2(xx.x), attn::ex2(xx.y));
    acc[k & 3] = __fadd2_rn(acc[k & 3], pp);
    p[k] = pack_half2(pp.x, pp.y);
  }
}

template <int DH, int G>
struct Cfg {
  static_assert(DH == 256, "d_h = 128 has its own kernel");
  static constexpr int TQ = BM / G;
  static constexpr int NCH = DH / 64;
  static constexpr int KGRP = 2;            // 64-channel chunks of K per barrier
  static constexpr int NKB = NCH / KGRP;    // K barriers
  // Q, one K tile and one V tile fill the 227 KB of shared memory; K is
  // released and refilled per KGRP 64-channel chunks (the S MMAs over them
  // are their only readers), V per half of its 128 keys (the PV MMAs of
  // that half).
  static constexpr uint32_t Q_BYTES = BM * DH * 2;
  static constexpr uint32_t KV_BYTES = BN * DH * 2;
  static constexpr uint32_t SMEM = Q_BYTES + 2 * KV_BYTES + 1024;
  static_assert(SMEM + 1536 + EPI_WARPS * 2048 <= 232448, "shared memory budget");
  // S buffers in TMEM (P lives in their first 64 columns): 0-127 and 128-255.
  static constexpr int NS = 2;
  static constexpr int LA = NS - 1;   // S issued this many tiles ahead of PV
  static __device__ __forceinline__ uint32_t s_col(int buf) {
    return static_cast<uint32_t>(buf) * 128u;
  }
};

using attn::Item;
using attn::decode_item;
using attn::ex2;
using attn::fmax3;

// Persistent: one CTA per SM walks the static order, or with `sched` the
// positions it takes from that counter (zeroed per launch).
// All pipeline phases count tiles (g) and items globally, so the K/V rings
// run ahead into the next item and the next item's Q is fetched as soon as
// the current item's last S MMA has consumed the Q buffer.
template <int DH, int G>
__global__ void __launch_bounds__(THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmK64,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    uint16_t* __restrict__ O, int o_f16,
                    const int32_t* __restrict__ pad_lens, int B, int T, int H, int H_kv,
                    int window, int num_q_tiles, int gsz, int num_items, unsigned int* sched,
                    int* status) {
  pdl_enter();
  using C = Cfg<DH, G>;
  // After a CTA of this or an earlier launch gave up, the rest do no work.
  if (*reinterpret_cast<volatile int*>(status) != 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + C::Q_BYTES;                    // 64-channel chunk c at c * CHUNK
  uint8_t* sV = sK + C::KV_BYTES;                     // key half h at c * CHUNK + h * CHUNK / 2
  __shared__ __align__(8) uint64_t q_full, q_empty, k_full[C::NKB], k_empty[C::NKB],
      v_full[2], v_empty[2], s_full[C::NS], p_full[2], pv_done[2], l_full[2],
      o_final, o_free, drain;
  // Row sums of O handed from the softmax to the epilogue, by item parity.
  __shared__ float lsum[2][BM];
  // Per epilogue warp: 32 rows x 32 O columns (64 B per row, 64-byte
  // swizzle) staged for a TMA store.
  __shared__ __align__(1024) uint8_t ostage[EPI_WARPS][32 * 64];
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_flag;
  __shared__ attn::SchedRing<SCHED_SLOTS, SCHED_CONSUMERS> ring;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&q_empty), 1);
    for (int s = 0; s < C::NKB; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 1);
    }
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&p_full[s]), SM_WARPS);
      mbar_init(smem_u32(&pv_done[s]), 1);
      mbar_init(smem_u32(&l_full[s]), SM_WARPS);
    }
    ring.init();
    mbar_init(smem_u32(&o_final), 1);
    mbar_init(smem_u32(&o_free), EPI_WARPS);
    mbar_init(smem_u32(&drain), 1);
    abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmK64);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_sh), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_sh;

  auto fetch_pos = [&](int rr) {
    return ring.fetch(rr, sched, num_items, &abort_flag, status, kSiteSchedEmpty);
  };
  auto take_pos = [&](int rr) {
    return ring.take(rr, sched, num_items, &abort_flag, status, kSiteSchedFull);
  };
  auto release_pos = [&](int rr) { ring.release(rr, sched); };

  // Registers move from the producer / MMA warpgroup to the softmax and
  // epilogue warpgroups (each warpgroup runs its setmaxnreg at the top of
  // its branch).
  if (warp < 4) {
    regs_decrease<REGS_LOW>();
    if (warp == 0) {
      if (lane == 0) {
        // ---------------- producer: Q of each item, then its K tiles chunk by chunk
        int f = 0, nq = 0;   // K tiles and Q tiles loaded
        int kf[C::NKB] = {};  // loads issued per K barrier
        bool ok = true;
        for (int rr = 0, pos; ok && (pos = fetch_pos(rr)) < num_items; ++rr) {
          const Item it = decode_item(pos, C::TQ, num_q_tiles, gsz, B, H_kv, T, window, pad_lens, true);
          if (it.pad) continue;
          // The Q buffer is free once the previous item's last S MMA is done.
          if (!mbar_wait(smem_u32(&q_empty), (nq & 1) ^ 1, &abort_flag, status, kSiteQ)) break;
          const uint32_t qb = smem_u32(&q_full);
          mbar_arrive_expect_tx(qb, C::Q_BYTES);
          for (int ch = 0; ch < C::NCH; ++ch)
            tma_load_4d(smem_u32(sQ + ch * CHUNK), &tmQ, qb, ch * 64, it.j * G, it.t0, it.b);
          ++nq;
          for (int i = 0; ok && i < it.n_tiles; ++i, ++f) {
            for (int kb = 0; kb < C::NKB; ++kb) {
              if (!mbar_wait(smem_u32(&k_empty[kb]), (f & 1) ^ 1, &abort_flag, status,
                             kSiteKEmpty)) {
                ok = false;
                break;
              }
              const uint32_t fb = smem_u32(&k_full[kb]);
              // The last tile's S reads only its first last_n keys: when they
              // fit in half a tile, only that half of each chunk is loaded.
              const bool half = i == it.n_tiles - 1 && it.last_n <= BN / 2;
              mbar_arrive_expect_tx(fb, half ? C::KGRP * CHUNK / 2 : C::KGRP * CHUNK);
              for (int ch = kb * C::KGRP; ch < (kb + 1) * C::KGRP; ++ch)
                tma_load_3d(smem_u32(sK + ch * CHUNK), half ? &tmK64 : &tmK, fb,
                            it.j * DH + ch * 64, it.s_base + i * BN, it.b);
              ++kf[kb];
            }
          }
        }
        if (nq > 0) mbar_wait_drain(smem_u32(&q_full), (nq - 1) & 1);
        for (int kb = 0; kb < C::NKB; ++kb)
          if (kf[kb] > 0) mbar_wait_drain(smem_u32(&k_full[kb]), (kf[kb] - 1) & 1);
      }
    } else if (warp == 2) {
      if (lane == 0) {
        // ---------------- producer: V tiles of each item, half by half
        int f = 0;            // V tiles loaded
        int vf[2] = {0, 0};   // loads issued per half
        bool ok = true;
        for (int rr = 0;; ++rr) {
          const int pos = take_pos(rr);
          release_pos(rr);
          if (pos >= num_items) break;
          const Item it = decode_item(pos, C::TQ, num_q_tiles, gsz, B, H_kv, T, window, pad_lens, true);
          for (int i = 0; ok && i < it.n_tiles; ++i, ++f) {
            for (int h = 0; h < 2; ++h) {
              if (!mbar_wait(smem_u32(&v_empty[h]), (f & 1) ^ 1, &abort_flag, status,
                             kSiteVEmpty)) {
                ok = false;
                break;
              }
              const uint32_t fb = smem_u32(&v_full[h]);
              if (h == 1 && i == it.n_tiles - 1 && it.last_n <= BN / 2) {
                // No row sees the second half of the last tile: nothing to load.
                mbar_arrive(fb);
              } else {
                mbar_arrive_expect_tx(fb, C::KV_BYTES / 2);
                for (int ch = 0; ch < C::NCH; ++ch)
                  tma_load_3d(smem_u32(sV + ch * CHUNK + h * (CHUNK / 2)), &tmV, fb,
                              it.j * DH + ch * 64, it.s_base + i * BN + h * (BN / 2), it.b);
              }
              ++vf[h];
            }
          }
          if (!ok) break;
        }
        for (int h = 0; h < 2; ++h)
          if (vf[h] > 0) mbar_wait_drain(smem_u32(&v_full[h]), (vf[h] - 1) & 1);
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer: the whole warp runs the loop (its state
      // warp-uniform); each tcgen05 instruction is issued by one elected lane.
      const uint32_t lead = elect_one();
      constexpr uint32_t idesc_qk = idesc_f16(BM, BN, /*f16*/ 0, 0, 0);
      constexpr uint32_t idesc_pv = idesc_f16(BM, DH, /*f16*/ 0, 0, /*B MN-major*/ 1);
      const uint32_t q_addr = smem_u32(sQ);
      int nitem = 0;   // items processed so far
      auto wait_all = [&](uint64_t& bar, int parity, int site) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar), parity, &abort_flag, status, site));
      };
      // PV of global tile gt, local tile lt of the current item, over its
      // first nk / 16 key steps (all 128 keys but on the item's last tile).
      auto issue_pv = [&](int gt, int lt, int nk) -> bool {
        // The first PV of an item overwrites O: the previous item's epilogue
        // must have read it.
        if (lt == 0 && nitem >= 1 && !wait_all(o_free, (nitem - 1) & 1, kSiteOFinal)) return false;
        if (!wait_all(p_full[gt & 1], (gt >> 1) & 1, kSitePFull)) return false;
        const uint32_t p_tmem = tbase + C::s_col(gt % C::NS);   // P over S_gt
        const uint32_t v_addr = smem_u32(sV);
        // Keys 64h .. 64h + 63 of V: its half h, released as soon as they are used.
        for (int h = 0; h < 2; ++h) {
          if (!wait_all(v_full[h], gt & 1, kSiteVFull)) return false;
          tc_fence_after();
#pragma unroll
          for (int k = 4 * h; k < 4 * h + 4; ++k)
            if (k * 16 < nk)
              mma_ts_lead(lead, tbase + O_COL, p_tmem + k * 8,
                          sdesc_sw128(v_addr + k * 2048, CHUNK, 1024), idesc_pv,
                          (lt > 0 || k > 0) ? 1u : 0u);
          mma_commit_lead(lead, smem_u32(&v_empty[h]));
        }
        mma_commit_lead(lead, smem_u32(&pv_done[gt & 1]));
        return true;
      };
      bool ok = true;
      int g = 0;
      for (int rr = 0; ok; ++rr) {
        int pos = take_pos(rr);
        pos = __shfl_sync(0xffffffffu, pos, 0);
        __syncwarp();
        if (lane == 0) release_pos(rr);
        if (pos >= num_items) break;
        const Item it = decode_item(pos, C::TQ, num_q_tiles, gsz, B, H_kv, T, window, pad_lens, true);
        if (it.pad) continue;
        if (!wait_all(q_full, nitem & 1, kSiteQ)) break;
        // The last tile's S covers only the keys some row can see.
        const uint32_t idesc_last = idesc_f16(BM, it.last_n, /*f16*/ 0, 0, 0);
        auto tile_keys = [&](int lt) { return lt == it.n_tiles - 1 ? it.last_n : BN; };
        for (int i = 0; ok && i < it.n_tiles; ++i, ++g) {
          // S buffer g % NS last held P_{g-NS}, whose PV this warp issued
          // before: the tensor pipe runs them in order.
          const int sb = g % C::NS;
          const uint32_t k_addr = smem_u32(sK);
          // Channels of K barrier kb (KGRP 64-channel chunks), released as soon
          // as their S MMAs have read them.
          for (int kb = 0; kb < C::NKB; ++kb) {
            if (!wait_all(k_full[kb], g & 1, kSiteKFull)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int k = 4 * C::KGRP * kb; k < 4 * C::KGRP * (kb + 1); ++k) {
              const uint32_t off = (k >> 2) * CHUNK + (k & 3) * 32;
              mma_ss_lead(lead, tbase + C::s_col(sb), sdesc_sw128(q_addr + off, 16, 1024),
                          sdesc_sw128(k_addr + off, 16, 1024),
                          i == it.n_tiles - 1 ? idesc_last : idesc_qk, k > 0 ? 1u : 0u);
            }
            mma_commit_lead(lead, smem_u32(&k_empty[kb]));
          }
          if (!ok) break;
          mma_commit_lead(lead, smem_u32(&s_full[sb]));
          if (i == it.n_tiles - 1) mma_commit_lead(lead, smem_u32(&q_empty));
          // S runs LA tiles ahead of PV (S_g reuses the buffer of P_{g-NS},
          // so LA <= NS - 1): the softmax finds the next S already computed.
          if (i >= C::LA && !issue_pv(g - C::LA, i - C::LA, tile_keys(i - C::LA))) {
            ok = false;
            break;
          }
        }
        // the PVs of the item's last LA tiles, then o_final: this item's O
        // accumulation is complete.
        for (int d = C::LA; ok && d >= 1; --d)
          if (it.n_tiles - d >= 0 && !issue_pv(g - d, it.n_tiles - d, tile_keys(it.n_tiles - d)))
            ok = false;
        if (!ok) break;
        mma_commit_lead(lead, smem_u32(&o_final));
        ++nitem;
      }
      mma_commit_lead(lead, smem_u32(&drain));
      mbar_wait_drain(smem_u32(&drain), 0);
    }
  } else if (warp < 8) {
    regs_increase<REGS_SOFT>();
    // ---------------- softmax: thread r owns row r of every S tile
    const int q = warp & 3;                // TMEM lane quarter (= warp % 4)
    const int r = q * 32 + lane;           // query row of this thread
    const int i_tok = r / G;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    int g = 0, nitem = 0;   // global tile, items
    bool ok = true;
    for (int rr = 0; ok; ++rr) {
      int pos = take_pos(rr);
      pos = __shfl_sync(0xffffffffu, pos, 0);
      __syncwarp();
      if (lane == 0) release_pos(rr);
      if (pos >= num_items) break;
      const Item it = decode_item(pos, C::TQ, num_q_tiles, gsz, B, H_kv, T, window, pad_lens, true);
      if (it.pad) continue;   // the epilogue writes its zero rows
      const int t = it.t0 + i_tok;
      const int kv_lo = window > 0 ? t - window + 1 : 0;   // keys kv_lo..kv_hi are kept
      const int kv_hi = min(t, it.valid - 1);
      float m_used = -INFINITY, l = 0.f;
      for (int i = 0; i < it.n_tiles; ++i, ++g) {
        const int sb = g % C::NS;
        const uint32_t s_base = tbase + lane_off + C::s_col(sb);
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&s_full[sb]), (g / C::NS) & 1,
                                               &abort_flag, status, kSiteSFull));
        if (!ok) break;
        tc_fence_after();
        const int s_tile = it.s_base + i * BN;
        const bool need_mask = (s_tile + BN - 1 > it.t0) || (s_tile + BN > it.valid) ||
                               (window > 0 && s_tile <= it.t_last - window);
        const int c_lo = kv_lo - s_tile, c_hi = kv_hi - s_tile;
        // The whole row of S in registers: four 32-column loads in flight
        // and one wait; their own max reduction gives the row max of an
        // unmasked tile.
        uint32_t ra[32], rb[32], rc[32], rd[32];
        float m0, m1, m2, m3;
        tmem_ld32_max(s_base, ra, m0);
        tmem_ld32_max(s_base + 32, rb, m1);
        tmem_ld32_max(s_base + 64, rc, m2);
        tmem_ld32_max(s_base + 96, rd, m3);
        tmem_ld_wait(ra);
        tmem_ld_wait(rb);
        tmem_ld_wait(rc);
        tmem_ld_wait(rd);
        tmem_ld_wait(m0);
        tmem_ld_wait(m1);
        tmem_ld_wait(m2);
        tmem_ld_wait(m3);
        float mx;
        if (!need_mask) {
          mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
        } else {
          // A 32-column chunk that every row of the warp sees whole keeps its
          // values and the TMEM load's max; the others are masked column by
          // column (a row's visible keys move by one every G rows, so most
          // chunks of a warp are whole).
#define G3_MASK_CHUNK(R, K, MK, OUT)                                              \
  {                                                                               \
    OUT = MK;                                                                     \
    if (!__all_sync(0xffffffffu, c_lo <= 32 * (K) && c_hi >= 32 * (K) + 31)) {   \
      mask32(R, 32 * (K) - c_lo, c_hi - c_lo);                                    \
      float a_ = -INFINITY, b_ = -INFINITY;                                       \
      _Pragma("unroll") for (int c = 0; c < 32; c += 2) {                         \
        a_ = fmaxf(a_, __uint_as_float(R[c]));                                    \
        b_ = fmaxf(b_, __uint_as_float(R[c + 1]));                                \
      }                                                                           \
      OUT = fmaxf(a_, b_);                                                        \
    }                                                                             \
  }
          float x0, x1, x2, x3;
          G3_MASK_CHUNK(ra, 0, m0, x0)
          G3_MASK_CHUNK(rb, 1, m1, x1)
          G3_MASK_CHUNK(rc, 2, m2, x2)
          G3_MASK_CHUNK(rd, 3, m3, x3)
#undef G3_MASK_CHUNK
          mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
        }
        mx *= LOG2E;
        const bool grow = mx > m_used + RESCALE_THRESHOLD;
        if (__any_sync(0xffffffffu, grow)) {
          const float m_new = grow ? mx : m_used;
          const float factor = (m_new == m_used) ? 1.f : ex2(m_used - m_new);
          if (i > 0) {
            // O holds this item's PV so far: rescale the row once the
            // previous PV has landed.
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&pv_done[(g - 1) & 1]),
                                                   ((g - 1) >> 1) & 1, &abort_flag, status,
                                                   kSiteORescale));
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < DH / 32; ++c) {
              uint32_t ro[32];
              const uint32_t ta = tbase + lane_off + O_COL + c * 32;
              tmem_ld32(ta, ro);
              tmem_ld_wait(ro);
#pragma unroll
              for (int e = 0; e < 32; ++e)
                ro[e] = __float_as_uint(__uint_as_float(ro[e]) * factor);
              tmem_st32(ta, ro);
            }
            tmem_st_wait();
          }
          l *= factor;
          m_used = m_new;
        }
        const float mref = (m_used == -INFINITY) ? 0.f : m_used;
        const float2 l2e = make_float2(LOG2E, LOG2E), negm = make_float2(-mref, -mref);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        // P of columns 0-63 goes over S columns 0-31, then P of columns
        // 64-127 over S columns 32-63: all of S is already in registers.
        {
          uint32_t p[32];
          exp_pack16(ra, p, acc, l2e, negm);
          exp_pack16(rb, p + 16, acc, l2e, negm);
          tmem_st32(s_base, p);
        }
        // Columns 64-127 of a last tile of at most 64 visible keys are all
        // masked (P = 0 there) and its PV stops at key 64: no exponentials.
        if (!(i == it.n_tiles - 1 && it.last_n <= BN / 2)) {
          uint32_t p[32];
          exp_pack16(rc, p, acc, l2e, negm);
          exp_pack16(rd, p + 16, acc, l2e, negm);
          tmem_st32(s_base + 32, p);
        }
        const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
        const float2 a = __fadd2_rn(a01, a23);
        l += a.x + a.y;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&p_full[g & 1]));
      }
      if (!ok) break;
      // The row sum goes to the epilogue; the softmax moves on to the next item.
      lsum[nitem & 1][r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&l_full[nitem & 1]));
      ++nitem;
    }
  } else {
    regs_decrease<REGS_EPI>();
    // ---------------- epilogue: column half eh of O for the CTA's 128 rows
    const int eh = (warp - 8) >> 2;
    const int q = warp & 3;                // TMEM lane quarter (= warp % 4)
    const int r = q * 32 + lane;
    const int t_off = r / G;
    const uint32_t o_base = tbase + (static_cast<uint32_t>(q * 32) << 16) + O_COL + eh * (DH / 2);
    uint8_t* stage = ostage[warp - 8];
    int nitem = 0;
    bool ok = true;
    for (int rr = 0; ok; ++rr) {
      int pos = take_pos(rr);
      pos = __shfl_sync(0xffffffffu, pos, 0);
      __syncwarp();
      if (lane == 0) release_pos(rr);
      if (pos >= num_items) break;
      const Item it = decode_item(pos, C::TQ, num_q_tiles, gsz, B, H_kv, T, window, pad_lens, true);
      if (it.pad) {
        // The whole tile is padding: its output rows are zero (bits 0 in bf16 and f16).
        const int rows = min(C::TQ, T - it.t0);
        const int vecs = rows * G * (DH / 8);
        for (int v = threadIdx.x - 256; v < vecs; v += EPI_WARPS * 32) {
          const int e = v * 8;
          const int c = e % DH, rg = e / DH;
          const int gg = rg % G, ii = rg / G;
          *reinterpret_cast<uint4*>(
              O + ((static_cast<size_t>(it.b) * T + it.t0 + ii) * H + it.j * G + gg) * DH + c) =
              make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      ok = __all_sync(0xffffffffu,
                      mbar_wait(smem_u32(&o_final), nitem & 1, &abort_flag, status, kSiteOFinal) &&
                          mbar_wait(smem_u32(&l_full[nitem & 1]), (nitem >> 1) & 1, &abort_flag,
                                    status, kSiteLFull));
      if (!ok) break;
      tc_fence_after();
      const bool row_valid = it.t0 + t_off < it.valid;
      const float l = lsum[nitem & 1][r];
      const float inv_l = row_valid && l > 0.f ? 1.f / l : 0.f;
      // This warp's 128 columns of its 32 rows, read two 32-column chunks at
      // a time and packed; then O is free for the next item's first PV.
      uint32_t pk[DH / 4];
#pragma unroll
      for (int c = 0; c < DH / 64; c += 2) {
        uint32_t ra[32], rb[32];
        tmem_ld32(o_base + c * 32, ra);
        tmem_ld32(o_base + c * 32 + 32, rb);
        tmem_ld_wait(ra);
        tmem_ld_wait(rb);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float a0 = __uint_as_float(ra[2 * e]) * inv_l;
          const float a1 = __uint_as_float(ra[2 * e + 1]) * inv_l;
          const float b0 = __uint_as_float(rb[2 * e]) * inv_l;
          const float b1 = __uint_as_float(rb[2 * e + 1]) * inv_l;
          pk[c * 16 + e] = o_f16 ? pack_half2(a0, a1) : pack_bf162(a0, a1);
          pk[c * 16 + 16 + e] = o_f16 ? pack_half2(b0, b1) : pack_bf162(b0, b1);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&o_free));
      // This warp's 32 rows are tokens t0 + 32q/G .. of the G heads: one box
      // {32 channels, G heads, 32/G tokens} of the [B, T, H, d_h] output per
      // chunk (rows past T are clipped by the store).
#pragma unroll
      for (int c = 0; c < DH / 64; ++c) {
        // The previous chunk's store must have read the staging tile.
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
        // row `lane` (64 B), 16-byte unit u at unit u ^ ((lane >> 1) & 3): 64-byte swizzle
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4*>(stage + lane * 64 + ((u ^ ((lane >> 1) & 3)) << 4)) =
              row_valid ? make_uint4(pk[c * 16 + 4 * u], pk[c * 16 + 4 * u + 1],
                                     pk[c * 16 + 4 * u + 2], pk[c * 16 + 4 * u + 3])
                        : make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_4d(&tmO, smem_u32(stage), eh * (DH / 2) + c * 32, it.j * G,
                       it.t0 + (q * 32) / G, it.b);
          bulk_commit_group();
        }
      }
      ++nitem;
    }
    if (lane == 0) bulk_wait_group_all();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int DH, int G>
cudaError_t launch_cfg(const void* Q, const void* K, const void* V, long ldkv, void* O,
                       int o_dtype, const int32_t* pad_lens, int B, int T, int H, int H_kv,
                       int window, unsigned int* sched, cudaStream_t stream, int* status,
                       bool sched_zeroed) {
  using C = Cfg<DH, G>;
  CUtensorMap tq, tk, tk64, tv;
  // Q' [B, T, H, d_h]: box {64 of d_h, the G heads of one group, TQ tokens, 1}.
  const uint64_t qdims[4] = {static_cast<uint64_t>(DH), static_cast<uint64_t>(H),
                             static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
  const uint64_t qstr[3] = {static_cast<uint64_t>(DH) * 2, static_cast<uint64_t>(H) * DH * 2,
                            static_cast<uint64_t>(T) * H * DH * 2};
  const uint32_t qbox[4] = {64, static_cast<uint32_t>(G), static_cast<uint32_t>(C::TQ), 1};
  // K', V: rows of a [B*T, ldkv] buffer; box {64 of d_h, 128 keys, 1}.
  const uint64_t kdims[3] = {static_cast<uint64_t>(H_kv) * DH, static_cast<uint64_t>(T),
                             static_cast<uint64_t>(B)};
  const uint64_t kstr[2] = {static_cast<uint64_t>(ldkv) * 2, static_cast<uint64_t>(T) * ldkv * 2};
  const uint32_t kbox[3] = {64, BN, 1};
  // V arrives half a tile of keys at a time; K in half tiles on an item's
  // last tile when no row sees past its first half.
  const uint32_t vbox[3] = {64, BN / 2, 1};
  // O [B, T, H, d_h] (16-bit, bf16 or fp16 bits alike): box {32 channels, G
  // heads, 32/G tokens, 1}, 64-byte swizzle.
  CUtensorMap to;
  const uint32_t obox[4] = {32, static_cast<uint32_t>(G), static_cast<uint32_t>(32 / G), 1};
  if (!encode_tiled(&to, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, O, qdims, qstr, obox,
                    CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  if (!encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, Q, qdims, qstr, qbox) ||
      !encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, K, kdims, kstr, kbox) ||
      !encode_tiled(&tk64, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, K, kdims, kstr, vbox) ||
      !encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, V, kdims, kstr, vbox))
    return cudaErrorInvalidValue;
  auto kern = attn_fwd_kernel<DH, G>;
  int launch_regs = 0;
  if (cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::SMEM, &launch_regs))
    return e;
  // The softmax and epilogue warpgroups' register increases wait for the
  // registers the producer / MMA warpgroup gives up: launch only when the
  // split fits the CTA's allocation.
  if (launch_regs * THREADS < REGS_SPLIT) return cudaErrorInvalidConfiguration;
  const int num_q_tiles = (T + C::TQ - 1) / C::TQ;
  const long items = static_cast<long>(num_q_tiles) * B * H_kv;
  if (items > 0x7fffffffL) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(items < num_sms() ? items : num_sms());
  const int gsz = attn::l2_group_size(B, H_kv, T, DH, window, C::TQ, grid);
  if (sched != nullptr && !sched_zeroed &&
      cudaMemsetAsync(sched, 0, sizeof(unsigned int), stream) != cudaSuccess)
    return cudaErrorUnknown;
  return launch_pdl(kern, dim3(grid), dim3(THREADS), C::SMEM, stream, tq, tk, tk64, tv, to,
                    static_cast<uint16_t*>(O), o_dtype == kF16 ? 1 : 0, pad_lens, B, T, H, H_kv,
                    window, num_q_tiles, gsz, static_cast<int>(items), sched, status);
}

}  // namespace

cudaError_t launch_flash_attention(const void* Q, const void* K, const void* V, long ldkv,
                                   void* O, int o_dtype, const int32_t* pad_lens, int B, int T,
                                   int H, int H_kv, int d_h, int window, void* sched,
                                   cudaStream_t stream, int* status, bool sched_zeroed) {
  if (B <= 0 || T <= 0) return cudaSuccess;
  if (o_dtype != kBF16 && o_dtype != kF16) return cudaErrorInvalidValue;
  if (d_h == 128)
    return launch_flash_attention_pair(Q, K, V, ldkv, O, o_dtype, pad_lens, B, T, H, H_kv, window,
                                       sched, stream, status, sched_zeroed);
  const int G = H / H_kv;
#define G3_ATTN_CASE(DH_, G_)                                                                   \
  if (d_h == DH_ && G == G_)                                                                    \
    return launch_cfg<DH_, G_>(Q, K, V, ldkv, O, o_dtype, pad_lens, B, T, H, H_kv, window,        \
                               static_cast<unsigned int*>(sched), stream, status, sched_zeroed);
  G3_ATTN_CASE(256, 1)
  G3_ATTN_CASE(256, 2)
  G3_ATTN_CASE(256, 4)
#undef G3_ATTN_CASE
  return cudaErrorInvalidValue;
}

}  // namespace g3
