// Flash-style attention forward for d_h = 128 with two query tiles per CTA
// ("Gemma 3 Attention Block", How it works: Scores and the GQA reshape).  It
// computes what attention.cu computes (same mask, padding, fp32 online
// softmax, fp16 operands, bf16/fp16 output); only the schedule differs.
//
// A work item is a pair of consecutive query tiles (2 x 128 rows; a tile is
// TQ = 128/G tokens x the G heads of kv head j) of one batch row, and both
// tiles stream the same K/V tiles of 128 keys.  Warps:
//   0      TMA: the pair's Q tiles, then the K ring
//   2      TMA: the V ring
//   1      TMEM allocation and MMA issue (the whole warp runs the loop,
//          one elected lane issues every tcgen05 instruction)
//   4-7    softmax of tile 0, 8-11 softmax of tile 1: one thread per row
//          holds all 128 columns of S in registers (setmaxnreg moves
//          registers to these warpgroups), so the two warpgroups never wait
//          for each other (no row-max exchange), and each rescales and
//          writes its own O.
// TMEM: S0 0-127, S1 128-255, O0 256-383, O1 384-511; P_e (fp16 pairs) is
// written over the first 64 columns of S_e.  The MMA issues S0_0, S1_0 and
// then, per KV tile i: PV0_i, S0_{i+1}, PV1_i, S1_{i+1}.  While one
// warpgroup computes its exponentials the tensor pipe runs the other tile's
// products; S_e of tile i+1 reuses S_e after PV_e of tile i, issued before it
// by the same warp (the tensor pipe runs them in order).
// Every wait is bounded (ptx.cuh); a free CTA takes the next item of the
// heavy-first order from the scheduler counter, as in attention.cu.
#include "attention_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace g3 {

namespace {

constexpr int DH = 128;
constexpr int NUM_WARPS = 12;
constexpr int THREADS = NUM_WARPS * 32;
constexpr int BM = 128;                 // query rows per tile
constexpr int BN = attn::KV_TILE;        // keys per KV tile
constexpr int SM_WARPS = 8;
constexpr int KS = 2, VS = 2;           // K / V ring depths
constexpr uint32_t CHUNK = 128 * 128;   // 128 rows x 64 elements (128 B), swizzled
constexpr uint32_t QT_BYTES = BM * DH * 2;      // one query tile
constexpr uint32_t KV_BYTES = BN * DH * 2;      // one K or V tile
constexpr uint32_t SMEM = 2 * QT_BYTES + (KS + VS) * KV_BYTES + 1024;
// TMEM columns of S_e (P_e over its first 64) and O_e.
__host__ __device__ constexpr uint32_t s_col(int e) { return static_cast<uint32_t>(e) * 128u; }
__host__ __device__ constexpr uint32_t o_col(int e) { return 256u + static_cast<uint32_t>(e) * 128u; }
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_THRESHOLD = 8.0f;   // log2 units
constexpr int SCHED_SLOTS = 4;
constexpr int SCHED_CONSUMERS = 2 + SM_WARPS;
static_assert(SMEM + 1024 <= 232448, "shared memory budget");
// Registers per thread: the launch gives every thread 65536 / 384 = 168;
// the producer / MMA warpgroup then drops to REGS_LOW and the two softmax
// warpgroups rise to REGS_HIGH (a whole 128-column row of S in registers).
constexpr int REGS_LAUNCH = 168;
constexpr int REGS_LOW = 96, REGS_HIGH = 200;
constexpr int REGS_SPLIT = 128 * REGS_LOW + 256 * REGS_HIGH;
static_assert(REGS_SPLIT <= THREADS * REGS_LAUNCH, "register split above the launch allocation");

enum : int {
  kSiteQ = 51, kSiteKEmpty, kSiteVEmpty, kSiteKFull, kSitePFull, kSiteVFull, kSiteSFull,
  kSiteORescale, kSiteOFinal, kSiteOFree, kSiteSchedFull, kSiteSchedEmpty
};

using attn::ex2;
using attn::fmax3;

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
    const float2 pp = make_float2(ex2(xx.x), ex2(xx.y));
    acc[k & 3] = __fadd2_rn(acc[k & 3], pp);
    p[k] = pack_half2(pp.x, pp.y);
  }
}

template <int G>
__global__ void __launch_bounds__(THREADS, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     uint16_t* __restrict__ O, int o_f16, const int32_t* __restrict__ pad_lens,
                     int B, int T, int H, int H_kv, int window, int num_pairs, int gsz,
                     int num_items, unsigned int* sched, int* status) {
  pdl_enter();
  constexpr int TQ = BM / G;
  if (*reinterpret_cast<volatile int*>(status) != 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                        // tile 0, tile 1
  uint8_t* sK = smem + 2 * QT_BYTES;         // KS stages
  uint8_t* sV = sK + KS * KV_BYTES;          // VS stages
  __shared__ __align__(8) uint64_t q_full, q_empty, k_full[KS], k_empty[KS], v_full[VS],
      v_empty[VS], s_full[2], p_full[2][2], o_final[2], o_free[2], drain;
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_flag;
  __shared__ attn::SchedRing<SCHED_SLOTS, SCHED_CONSUMERS> ring;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&q_empty), 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 1);
    }
    for (int e = 0; e < 2; ++e) {
      mbar_init(smem_u32(&s_full[e]), 1);
      mbar_init(smem_u32(&o_final[e]), 1);
      mbar_init(smem_u32(&o_free[e]), 4);
      for (int s = 0; s < 2; ++s) {
        mbar_init(smem_u32(&p_full[e][s]), 4);
      }
    }
    ring.init();
    mbar_init(smem_u32(&drain), 1);
    abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
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

  // Registers move from the producer / MMA warpgroup to the softmax warpgroups
  // (each warpgroup executes its own setmaxnreg at the top of its branch).
  if (warp < 4) {
    regs_decrease<REGS_LOW>();
    if (warp == 0) {
      if (lane == 0) {
        // ---------------- producer: the pair's Q tiles, then its K tiles
        int fills[KS] = {};
        int f = 0, nq = 0;
        bool ok = true;
        for (int rr = 0, pos; ok && (pos = fetch_pos(rr)) < num_items; ++rr) {
          const attn::Item it =
            attn::decode_item(pos, 2 * TQ, num_pairs, gsz, B, H_kv, T, window, pad_lens);
          if (it.pad) continue;
          if (!mbar_wait(smem_u32(&q_empty), (nq & 1) ^ 1, &abort_flag, status, kSiteQ)) break;
          const uint32_t qb = smem_u32(&q_full);
          mbar_arrive_expect_tx(qb, 2 * QT_BYTES);
          for (int e = 0; e < 2; ++e)
            for (int ch = 0; ch < DH / 64; ++ch)
              tma_load_4d(smem_u32(sQ + e * QT_BYTES + ch * CHUNK), &tmQ, qb, ch * 64, it.j * G,
                          it.t0 + e * TQ, it.b);
          ++nq;
          for (int i = 0; i < it.n_tiles; ++i, ++f) {
            const int st = f % KS;
            if (!mbar_wait(smem_u32(&k_empty[st]), ((f / KS) & 1) ^ 1, &abort_flag, status,
                           kSiteKEmpty)) {
              ok = false;
              break;
            }
            const uint32_t fb = smem_u32(&k_full[st]);
            mbar_arrive_expect_tx(fb, KV_BYTES);
            for (int ch = 0; ch < DH / 64; ++ch)
              tma_load_3d(smem_u32(sK + st * KV_BYTES + ch * CHUNK), &tmK, fb, it.j * DH + ch * 64,
                          (it.tile_lo + i) * BN, it.b);
            ++fills[st];
          }
        }
        if (nq > 0) mbar_wait_drain(smem_u32(&q_full), (nq - 1) & 1);
        for (int s = 0; s < KS; ++s)
          if (fills[s] > 0) mbar_wait_drain(smem_u32(&k_full[s]), (fills[s] - 1) & 1);
      }
    } else if (warp == 2) {
      if (lane == 0) {
        // ---------------- producer: V tiles
        int fills[VS] = {};
        int f = 0;
        bool ok = true;
        for (int rr = 0;; ++rr) {
          const int pos = take_pos(rr);
          release_pos(rr);
          if (pos >= num_items) break;
          const attn::Item it =
            attn::decode_item(pos, 2 * TQ, num_pairs, gsz, B, H_kv, T, window, pad_lens);
          for (int i = 0; i < it.n_tiles; ++i, ++f) {
            const int st = f % VS;
            if (!mbar_wait(smem_u32(&v_empty[st]), ((f / VS) & 1) ^ 1, &abort_flag, status,
                           kSiteVEmpty)) {
              ok = false;
              break;
            }
            const uint32_t fb = smem_u32(&v_full[st]);
            mbar_arrive_expect_tx(fb, KV_BYTES);
            for (int ch = 0; ch < DH / 64; ++ch)
              tma_load_3d(smem_u32(sV + st * KV_BYTES + ch * CHUNK), &tmV, fb, it.j * DH + ch * 64,
                          (it.tile_lo + i) * BN, it.b);
            ++fills[st];
          }
          if (!ok) break;
        }
        for (int s = 0; s < VS; ++s)
          if (fills[s] > 0) mbar_wait_drain(smem_u32(&v_full[s]), (fills[s] - 1) & 1);
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer: the whole warp runs the loop (its state
      // warp-uniform); each tcgen05 instruction is issued by one elected lane.
      constexpr uint32_t idesc_qk = idesc_f16(BM, BN, /*f16*/ 0, 0, 0);
      constexpr uint32_t idesc_pv = idesc_f16(BM, DH, /*f16*/ 0, 0, /*B MN-major*/ 1);
      const uint32_t lead = elect_one();   // the lane that issues every tcgen05 instruction
      int nitem = 0;
      int g0 = 0;   // global index of the current item's first tile
      auto wait_all = [&](uint64_t& bar, int parity, int site) -> bool {
        return __all_sync(0xffffffffu,
                          mbar_wait(smem_u32(&bar), parity, &abort_flag, status, site));
      };
      // S_e of global tile g from K stage g % KS.
      auto issue_s = [&](int e, int g) {
        const uint32_t q_addr = smem_u32(sQ + e * QT_BYTES);
        const uint32_t k_addr = smem_u32(sK + (g % KS) * KV_BYTES);
#pragma unroll
        for (int k = 0; k < DH / 16; ++k) {
          const uint32_t off = (k >> 2) * CHUNK + (k & 3) * 32;
          mma_ss_lead(lead, tbase + s_col(e), sdesc_sw128(q_addr + off, 16, 1024),
                      sdesc_sw128(k_addr + off, 16, 1024), idesc_qk, k > 0 ? 1u : 0u);
        }
        mma_commit_lead(lead, smem_u32(&s_full[e]));
      };
      // PV_e of global tile g, item-local tile i.
      auto issue_pv = [&](int e, int g, int i) -> bool {
        if (i == 0 && nitem >= 1 && !wait_all(o_free[e], (nitem - 1) & 1, kSiteOFree)) return false;
        if (!wait_all(p_full[e][g & 1], (g >> 1) & 1, kSitePFull)) return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(sV + (g % VS) * KV_BYTES);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ts_lead(lead, tbase + o_col(e), tbase + s_col(e) + k * 8,
                      sdesc_sw128(v_addr + k * 2048, CHUNK, 1024), idesc_pv,
                      (i > 0 || k > 0) ? 1u : 0u);
        return true;
      };
      bool ok = true;
      for (int rr = 0; ok; ++rr) {
        int pos = take_pos(rr);
        pos = __shfl_sync(0xffffffffu, pos, 0);
        __syncwarp();
        if (lane == 0) release_pos(rr);
        if (pos >= num_items) break;
        const attn::Item it =
            attn::decode_item(pos, 2 * TQ, num_pairs, gsz, B, H_kv, T, window, pad_lens);
        if (it.pad) continue;
        const int n = it.n_tiles;
        if (!wait_all(q_full, nitem & 1, kSiteQ) ||
            !wait_all(k_full[g0 % KS], (g0 / KS) & 1, kSiteKFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(0, g0);
        issue_s(1, g0);
        mma_commit_lead(lead, smem_u32(&k_empty[g0 % KS]));
        if (n == 1) mma_commit_lead(lead, smem_u32(&q_empty));
        for (int i = 0; i < n; ++i) {
          const int g = g0 + i;
          if (!wait_all(v_full[g % VS], (g / VS) & 1, kSiteVFull) || !issue_pv(0, g, i)) {
            ok = false;
            break;
          }
          if (i + 1 < n) {
            if (!wait_all(k_full[(g + 1) % KS], ((g + 1) / KS) & 1, kSiteKFull)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(0, g + 1);
          }
          if (i + 1 == n) mma_commit_lead(lead, smem_u32(&o_final[0]));   // O0 of this item complete
          if (!issue_pv(1, g, i)) {
            ok = false;
            break;
          }
          mma_commit_lead(lead, smem_u32(&v_empty[g % VS]));
          if (i + 1 < n) {
            issue_s(1, g + 1);
            mma_commit_lead(lead, smem_u32(&k_empty[(g + 1) % KS]));
            if (i + 1 == n - 1) mma_commit_lead(lead, smem_u32(&q_empty));
          } else {
            mma_commit_lead(lead, smem_u32(&o_final[1]));
          }
        }
        if (!ok) break;
        g0 += n;
        ++nitem;
      }
      mma_commit_lead(lead, smem_u32(&drain));
      mbar_wait_drain(smem_u32(&drain), 0);
    }
  } else {
    regs_increase<REGS_HIGH>();
    // ---------------- softmax of query tile e, then its epilogue
    const int e = (warp - 4) >> 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;          // row of the tile
    const int i_tok = r / G;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t s_base = tbase + lane_off + s_col(e);
    const uint32_t o_base = tbase + lane_off + o_col(e);
    int g0 = 0, nitem = 0;
    bool ok = true;
    for (int rr = 0; ok; ++rr) {
      int pos = take_pos(rr);
      pos = __shfl_sync(0xffffffffu, pos, 0);
      __syncwarp();
      if (lane == 0) release_pos(rr);
      if (pos >= num_items) break;
      const attn::Item it =
            attn::decode_item(pos, 2 * TQ, num_pairs, gsz, B, H_kv, T, window, pad_lens);
      const int te0 = it.t0 + e * TQ;       // first token of this tile
      if (it.pad) {
        // The whole pair is padding: rows < T of this tile are zero.
        const int rows = max(0, min(TQ, T - te0));
        const int vecs = rows * G * (DH / 8);
        for (int v = (threadIdx.x - 128) & 127; v < vecs; v += 128) {
          const int el = v * 8;
          const int c = el % DH, rg = el / DH;
          const int gg = rg % G, ii = rg / G;
          *reinterpret_cast<uint4*>(
              O + ((static_cast<size_t>(it.b) * T + te0 + ii) * H + it.j * G + gg) * DH + c) =
              make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int t = te0 + i_tok;
      const int kv_lo = window > 0 ? t - window + 1 : 0;   // keys kv_lo..kv_hi are kept
      const int kv_hi = min(t, it.valid - 1);
      const int t_last_e = min(te0 + TQ, it.valid) - 1;  // < te0 when the tile is all padding
      float m_used = -INFINITY, l = 0.f;
      for (int i = 0; i < it.n_tiles; ++i) {
        const int g = g0 + i;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&s_full[e]), g & 1, &abort_flag, status,
                                               kSiteSFull));
        if (!ok) break;
        tc_fence_after();
        const int s_tile = (it.tile_lo + i) * BN;
        const bool need_mask = (s_tile + BN - 1 > te0) || (s_tile + BN > it.valid) ||
                               t_last_e < te0 || (window > 0 && s_tile <= t_last_e - window);
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
          mask32(ra, 0 - c_lo, c_hi - c_lo);
          mask32(rb, 32 - c_lo, c_hi - c_lo);
          mask32(rc, 64 - c_lo, c_hi - c_lo);
          mask32(rd, 96 - c_lo, c_hi - c_lo);
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < 32; ++c)
            m4[c & 3] = fmax3(m4[c & 3],
                              fmax3(__uint_as_float(ra[c]), __uint_as_float(rb[c]),
                                    __uint_as_float(rc[c])),
                              __uint_as_float(rd[c]));
          mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        mx *= LOG2E;
        const bool grow = mx > m_used + RESCALE_THRESHOLD;
        if (__any_sync(0xffffffffu, grow)) {
          const float m_new = grow ? mx : m_used;
          const float factor = (m_new == m_used) ? 1.f : ex2(m_used - m_new);
          if (i > 0) {
            // O_e holds this item's PV so far.  The previous PV_e has landed:
            // S_e of this tile, whose completion the s_full wait above saw,
            // was committed after that PV_e was issued.
#pragma unroll 1
            for (int c = 0; c < DH / 32; ++c) {
              uint32_t ro[32];
              tmem_ld32(o_base + c * 32, ro);
              tmem_ld_wait(ro);
#pragma unroll
              for (int k = 0; k < 32; ++k)
                ro[k] = __float_as_uint(__uint_as_float(ro[k]) * factor);
              tmem_st32(o_base + c * 32, ro);
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
        {
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
        if (lane == 0) mbar_arrive(smem_u32(&p_full[e][g & 1]));
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&o_final[e]), nitem & 1, &abort_flag,
                                             status, kSiteOFinal));
      if (!ok) break;
      tc_fence_after();
      const bool row_valid = t < it.valid;
      const float inv_l = row_valid && l > 0.f ? 1.f / l : 0.f;
      // Each thread writes its own row of O_e straight from registers
      // (16-byte stores); rows past T, in a second tile beyond the sequence,
      // are not written.
      {
        uint32_t ra[32], rb[32], rc[32], rd[32];
        tmem_ld32(o_base, ra);
        tmem_ld32(o_base + 32, rb);
        tmem_ld32(o_base + 64, rc);
        tmem_ld32(o_base + 96, rd);
        tmem_ld_wait(ra);
        tmem_ld_wait(rb);
        tmem_ld_wait(rc);
        tmem_ld_wait(rd);
        // O_e has been read: the next item's first PV_e may overwrite it.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&o_free[e]));
        if (t < T) {
          uint16_t* orow =
              O + ((static_cast<size_t>(it.b) * T + t) * H + it.j * G + r % G) * DH;
          store_row32(orow, ra, inv_l, row_valid, o_f16);
          store_row32(orow + 32, rb, inv_l, row_valid, o_f16);
          store_row32(orow + 64, rc, inv_l, row_valid, o_f16);
          store_row32(orow + 96, rd, inv_l, row_valid, o_f16);
        }
      }
      g0 += it.n_tiles;
      ++nitem;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int G>
cudaError_t launch_pair_cfg(const void* Q, const void* K, const void* V, long ldkv, void* O,
                            int o_dtype, const int32_t* pad_lens, int B, int T, int H, int H_kv,
                            int window, unsigned int* sched, cudaStream_t stream, int* status,
                            bool sched_zeroed) {
  constexpr int TQ = BM / G;
  CUtensorMap tq, tk, tv;
  const uint64_t qdims[4] = {static_cast<uint64_t>(DH), static_cast<uint64_t>(H),
                             static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
  const uint64_t qstr[3] = {static_cast<uint64_t>(DH) * 2, static_cast<uint64_t>(H) * DH * 2,
                            static_cast<uint64_t>(T) * H * DH * 2};
  const uint32_t qbox[4] = {64, static_cast<uint32_t>(G), static_cast<uint32_t>(TQ), 1};
  const uint64_t kdims[3] = {static_cast<uint64_t>(H_kv) * DH, static_cast<uint64_t>(T),
                             static_cast<uint64_t>(B)};
  const uint64_t kstr[2] = {static_cast<uint64_t>(ldkv) * 2, static_cast<uint64_t>(T) * ldkv * 2};
  const uint32_t kbox[3] = {64, BN, 1};
  // O [B, T, H, d_h] is written with 16-byte stores.
  if (reinterpret_cast<uintptr_t>(O) % 16 != 0) return cudaErrorInvalidValue;
  if (!encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, Q, qdims, qstr, qbox) ||
      !encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, K, kdims, kstr, kbox) ||
      !encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, V, kdims, kstr, kbox))
    return cudaErrorInvalidValue;
  auto kern = attn_pair_kernel<G>;
  int launch_regs = 0;
  if (cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), SMEM, &launch_regs))
    return e;
  // The softmax warpgroups' register increase waits for the registers the
  // other warpgroup gives up: launch only when the split fits the CTA's
  // allocation.
  if (launch_regs * THREADS < REGS_SPLIT) return cudaErrorInvalidConfiguration;
  const int num_pairs = (T + 2 * TQ - 1) / (2 * TQ);
  const long items = static_cast<long>(num_pairs) * B * H_kv;
  if (items > 0x7fffffffL) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(items < num_sms() ? items : num_sms());
  const int gsz = attn::l2_group_size(B, H_kv, T, DH, window, 2 * TQ, grid);
  if (sched != nullptr && !sched_zeroed &&
      cudaMemsetAsync(sched, 0, sizeof(unsigned int), stream) != cudaSuccess)
    return cudaErrorUnknown;
  return launch_pdl(kern, dim3(grid), dim3(THREADS), SMEM, stream, tq, tk, tv,
                    static_cast<uint16_t*>(O), o_dtype == kF16 ? 1 : 0, pad_lens, B, T, H, H_kv,
                    window, num_pairs, gsz, static_cast<int>(items), sched, status);
}

}  // namespace

cudaError_t launch_flash_attention_pair(const void* Q, const void* K, const void* V, long ldkv,
                                        void* O, int o_dtype, const int32_t* pad_lens, int B,
                                        int T, int H, int H_kv, int window, void* sched,
                                        cudaStream_t stream, int* status, bool sched_zeroed) {
  const int G = H / H_kv;
  unsigned int* sc = static_cast<unsigned int*>(sched);
  if (G == 1)
    return launch_pair_cfg<1>(Q, K, V, ldkv, O, o_dtype, pad_lens, B, T, H, H_kv, window, sc,
                              stream, status, sched_zeroed);
  if (G == 2)
    return launch_pair_cfg<2>(Q, K, V, ldkv, O, o_dtype, pad_lens, B, T, H, H_kv, window, sc,
                              stream, status, sched_zeroed);
  if (G == 4)
    return launch_pair_cfg<4>(Q, K, V, ldkv, O, o_dtype, pad_lens, B, T, H, H_kv, window, sc,
                              stream, status, sched_zeroed);
  return cudaErrorInvalidValue;
}

}  // namespace g3
