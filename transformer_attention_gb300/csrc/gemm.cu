// Projection GEMM on the 5th-generation tensor cores (tcgen05).
//
// C[M,N] = A[M,K] * W[N,K]^T with bf16 (or fp16) operands and fp32
// accumulation: the Q / KV projections (x against Wq, Wkv) and the output
// projection (O against Wo) of the attention layer ("Gemma 3 Attention
// Block", How it works: Projections and the attn_vec_einsum).
//
// Design (one CTA per SM, persistent), for tiles of 128 x 256 ("one half"):
//   warp 0      TMA producer: 128x64 A and 256x64 W tiles, 128-byte swizzle,
//               into a 4-stage shared-memory ring (48 KB per stage).
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma
//               (M=128, N=256, K=16): the whole warp runs the loop, one
//               elected lane issues each instruction; accumulators live in
//               TMEM, double-buffered (2 x 256 columns) so the epilogue of one
//               tile overlaps the main loop of the next.
//   warps 4-7   epilogue: tcgen05.ld of the accumulator rows (one TMEM lane
//               per thread), conversion to the output type, then each warp
//               writes its 32 rows x 128 B chunk into a double-buffered,
//               128-byte-swizzled shared-memory staging tile that one lane
//               stores with a TMA bulk tensor store (full-line writes instead
//               of 32 scattered 16-byte pieces per warp instruction).
// Tiles of 256 x 256 ("two halves", plain outputs of large launches): each
// stage holds two 128-row A tiles and one W tile (64 KB, 3 stages), both
// halves' MMAs read the same W tile, and the halves' accumulators fill TMEM
// (half h at column 256 h).  The epilogue drains half 0, then half 1; the
// next tile's half-0 MMAs start as soon as half 0 is drained and its half-1
// MMAs catch up on the held stages once half 1 is (the MMA issuer polls).
// Both halves sum their k-steps in the same order as a one-half tile, so
// the output is the same bit for bit.
// Tiles are visited in groups of consecutive M tiles (N-tiles varying slowest
// within a group, in reverse on odd groups), so the tiles in flight share A
// rows and W rows through L2; weights larger than L2 get groups of ~20 MB of
// A.  Given the batch rows' trailing padding, M tiles of pad rows alone are
// left out of that order (their rows are never read by the attention; the
// epilogue writes zeros from a given column on where a later kernel reads
// them).
// Epilogue modes: plain conversion; GeGLU (the feed-forward gating
// projection); and the attention prologue ("QK-Norm", How it works; "Gemma 3
// Attention Block", How it works: QK-norm, then RoPE, then scale) applied to
// the Q or K head vectors straight from the fp32 accumulator: a 256-wide tile
// holds one d_h = 256 head or two d_h = 128 heads of a row, so each thread
// (one row) sums the squares of its head, then rotates the pairs (c, c +
// d_h/2) with (1 + gamma) and the query scale folded in.
// Every mbarrier wait is bounded (see ptx.cuh).
#include <atomic>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace g3 {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, THREADS = 256;
constexpr uint32_t A_BYTES = BM * BK * 2;   // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;   // 32 KB
constexpr uint32_t STAGING_BYTES = 32 * 128;           // one warp's 32 rows x 128 B
constexpr uint32_t STAGING_TOTAL = 4 * 2 * STAGING_BYTES;   // 4 warps, double-buffered
// A tile is HALVES x 128 rows by 256 columns.  HALVES = 1: a stage holds one
// A tile and one W tile (48 KB, four stages) and the accumulator is
// double-buffered in TMEM.  HALVES = 2: a stage holds two A tiles and one W
// tile (64 KB, three stages) and the two 128-row halves' accumulators fill
// TMEM; each W byte brought into shared memory then feeds twice the MMA
// work.  Measured on GB300 with the whole main loop issued twice per stage
// (half the shared-memory fill per FLOP): the 4B and 27B projections ran at
// an effective 2130-2140 TF/s against 1670-1690, so the one-tile main loop
// waits on its operand copies rather than on the tensor core.
template <int HALVES>
struct Ring {
  static constexpr int STAGES = HALVES == 2 ? 3 : 4;
  static constexpr uint32_t STAGE_BYTES = HALVES * A_BYTES + B_BYTES;
  static constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_TOTAL + 1024;
};
static_assert(Ring<2>::SMEM_BYTES + 1024 <= 232448, "two-half ring exceeds shared memory");
// Rasterisation: tiles are visited in groups of consecutive M tiles, the N
// tile varying slowest within a group, so a group's A rows stay in L2 while
// W streams past them.  A weight that fits in L2 (up to kSmallWeightBytes)
// is read from DRAM once whatever the grouping, and groups of 8 M tiles keep
// each A tile shared by many CTAs at once.  A larger weight is read once per
// group, so its groups hold about kGroupBytes of A.  Measured on GB300 (27B
// projections, W 44-88 MB): 8-tile groups 1570, ~20 MB groups 1644, ~40 MB
// 1624, ~80 MB 1494 TF/s; on the 1B shapes (W 3.5 MB) 8-tile groups were
// the fastest (1250 against 1173 TF/s with ~20 MB groups).
constexpr int kSmallGroupM = 8;
constexpr size_t kSmallWeightBytes = size_t(32) << 20;
constexpr size_t kGroupBytes = size_t(20) << 20;

// Unit t of the grouped order -> (m unit, n tile); a group spans `group`
// m units.  Odd groups walk the N tiles in reverse, so each group starts on
// the W tiles the previous one used last, which are still in L2 (a weight
// larger than L2 is otherwise read from DRAM once per group in full).
__device__ __forceinline__ void tile_coords(int t, int m_units, int n_tiles, int group, int& mu,
                                            int& nt) {
  const int per_group = group * n_tiles;
  const int g = t / per_group;
  const int first_m = g * group;
  const int gm = min(group, m_units - first_m);
  const int r = t % per_group;
  mu = first_m + r % gm;
  nt = (g & 1) ? n_tiles - 1 - r / gm : r / gm;
}
constexpr uint32_t TMEM_COLS = 512;
constexpr int kMaxPadSegs = 64;   // batch segments whose pad-only M tiles are skipped

enum : int { kSiteEmpty = 1, kSiteFull = 2, kSiteAccEmpty = 3, kSiteAccFull = 4 };

enum : int { kEpiPlain = 0, kEpiGeglu = 1, kEpiQkNorm = 2 };

// Arguments of the QK-norm + RoPE epilogue: columns [0, n_norm) of C are head
// vectors (d_h each) to normalise with (1 + gamma), rotate at pos[row] and
// multiply by scale; columns from n_norm on are converted as they are.
// n1 > 0 splits the output columns in two segments with their own weight
// and output maps (tmB2 / tmC2 for columns n1..): the Q projection (segment
// 0, gamma / scale / n_norm) and the KV projection (segment 1, gamma2 /
// scale2 / n_norm2, counted from the segment's first column) in one launch,
// so each tile of x feeds both.
struct QkEpi {
  RopeFreqs freqs;
  const __nv_bfloat16* gamma;
  const __nv_bfloat16* gamma2;
  const int32_t* pos;
  int n_norm, n_norm2, n1;
  float scale, scale2;
};

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  return pack_half2(a, b);
}
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  return pack_bf162(a, b);
}

// GeGLU epilogue of the feed-forward gating projection ("Full Gemma 3
// Block", How it works: MLP): z = GELU(g) * u with the tanh-form GELU
// 0.5 g (1 + tanh t), t = sqrt(2/pi) (g + 0.044715 g^3).  Since
// 0.5 (1 + tanh t) = 1 / (1 + exp(-2 t)), it is evaluated as
// g u / (1 + exp(-2 t)) with the hardware exponential and division (one
// approximate exp2 and one reciprocal; relative error ~1e-6, against fp16's
// 5e-4 of the stored z).  Large negative t gives exp = inf and z = 0, the
// function's limit.
__device__ __forceinline__ float gelu_tanh_mul(float g, float u) {
  const float kM2C = -1.5957691216057308f;   // -2 sqrt(2 / pi)
  const float e = __expf(kM2C * fmaf(0.044715f * g, g * g, g));
  return __fdividef(g * u, 1.f + e);
}

// GEGLU = false: C[M,N] = A W^T.  GEGLU = true: W is the [2*N, K] gating
// weight (rows [0, N) gate, [N, 2N) up); each 256-wide accumulator tile holds
// 128 gate and the matching 128 up columns, and the epilogue writes
// C[M, N] = GELU(A Wg^T) * (A Wu^T).
// EPI = kEpiQkNorm (OutT = __half, DH = d_h): the attention prologue above.
// HALVES: 128-row halves per tile (Ring).
template <int AB_BF16, typename OutT, int EPI, int DH, bool PAD, int HALVES>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ CUtensorMap tmC2, int M, int N, int K, int group_m,
                   const int32_t* __restrict__ pad_lens, int seg_T, int zero_from, int* status,
                   const __grid_constant__ QkEpi epi) {
  pdl_enter();
  constexpr bool GEGLU = EPI == kEpiGeglu;
  static_assert(EPI != kEpiQkNorm || (std::is_same<OutT, __half>::value && (DH == 128 || DH == 256)),
                "the QK-norm epilogue writes fp16 head vectors of 128 or 256");
  // The fused prologue's epilogue is as long as a short main loop, which two
  // halves sharing TMEM could not hide: it keeps one-half tiles.
  static_assert(HALVES == 1 || (HALVES == 2 && EPI != kEpiQkNorm), "two halves: plain or GeGLU");
  constexpr int STAGES = Ring<HALVES>::STAGES;
  constexpr uint32_t STAGE_BYTES = Ring<HALVES>::STAGE_BYTES;
  constexpr int BN_OUT = GEGLU ? BN / 2 : BN;   // output columns per tile
  constexpr int CW = 128 / static_cast<int>(sizeof(OutT));   // output columns per 128 B chunk
  // A kernel launched after an earlier one gave up does no work.
  if (*reinterpret_cast<volatile int*>(status) != 0) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ __align__(8) uint64_t accf_bar[2], acce_bar[2], drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (M + BM - 1) / BM, n_tiles = (N + BN_OUT - 1) / BN_OUT;
  const int unit0 = blockIdx.x, unit_step = gridDim.x;
  const int num_kb = (K + BK - 1) / BK;
  // Rows of batch segments of seg_T rows with trailing padding (pad_lens):
  // M tiles holding only pad rows are not computed; after the computed tiles
  // the epilogue writes zeros in their N tiles from column zero_from on (a
  // multiple of the tile width; N or more: none).  pre_ne[b] / pre_z[b]:
  // computed / pad-only M tiles of the segments before b.
  __shared__ int pre_ne[kMaxPadSegs + 1], pre_z[kMaxPadSegs + 1];
  const int n_seg = seg_T > 0 ? M / seg_T : 0;
  // (PAD false: an instantiation for calls without padding information, in
  // which all of this folds away)
  const bool skip = PAD && pad_lens != nullptr && seg_T > 0 && seg_T % BM == 0 &&
                    M % seg_T == 0 && n_seg <= kMaxPadSegs;
  const int seg_tiles = skip ? seg_T / BM : 0;
  if (skip && warp == 2) {
    // Warp 2 (idle in this kernel) while warp 1 allocates TMEM: its lanes
    // load 32 segments' pad counts at once and a warp scan forms the prefixes.
    if (lane == 0) pre_ne[0] = pre_z[0] = 0;
    int carry_ne = 0, carry_z = 0;
    for (int b0 = 0; b0 < n_seg; b0 += 32) {
      const int b = b0 + lane;
      int ne = 0, z = 0;
      if (b < n_seg) {
        const int valid = min(max(seg_T - pad_lens[b], 0), seg_T);
        ne = (valid + BM - 1) / BM;
        z = seg_tiles - ne;
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, ne, o);
        const int c = __shfl_up_sync(0xffffffffu, z, o);
        if (lane >= o) {
          ne += a;
          z += c;
        }
      }
      if (b < n_seg) {
        pre_ne[b + 1] = carry_ne + ne;
        pre_z[b + 1] = carry_z + z;
      }
      carry_ne += __shfl_sync(0xffffffffu, ne, 31);
      carry_z += __shfl_sync(0xffffffffu, z, 31);
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&accf_bar[b]), 1);
      mbar_init(smem_u32(&acce_bar[b]), 4);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    if (epi.n1 > 0) {
      tma_prefetch_desc(&tmB2);
      tma_prefetch_desc(&tmC2);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), TMEM_COLS);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_sh;
  const int m_units = skip ? pre_ne[n_seg] : m_tiles;   // computed 128-row M tiles
  const int z_tiles = skip ? pre_z[n_seg] : 0;           // pad-only M tiles
  const int mu_units = (m_units + HALVES - 1) / HALVES;  // tile rows of HALVES of them
  const int num_units = mu_units * n_tiles;
  const int zn0 = zero_from < N ? zero_from / BN_OUT : n_tiles;   // first zeroed N tile
  const int zero_units = z_tiles * (n_tiles - zn0);
  // unit u -> the M tile of each half (-1: past the last computed tile) and
  // the N tile
  auto unit_coords = [&](int u, int (&mt)[HALVES], int& nt) {
    int cu;
    tile_coords(u, mu_units, n_tiles, group_m, cu, nt);
#pragma unroll
    for (int h = 0; h < HALVES; ++h) {
      int cm = cu * HALVES + h;
      if (cm >= m_units) {
        mt[h] = -1;
        continue;
      }
      if (skip) {
        int b = 0;
        while (pre_ne[b + 1] <= cm) ++b;
        cm = b * seg_tiles + (cm - pre_ne[b]);
      }
      mt[h] = cm;
    }
  };
  // zero unit z -> (pad-only M tile, N tile)
  auto zero_coords = [&](int z, int& mt, int& nt) {
    const int zt = z_tiles > 0 ? z_tiles : 1;   // (no zero units without pad-only tiles)
    const int zm = z % zt;
    nt = zn0 + z / zt;
    int b = 0;
    while (pre_z[b + 1] <= zm) ++b;
    mt = b * seg_tiles + (pre_ne[b + 1] - pre_ne[b]) + (zm - pre_z[b]);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      int fills[STAGES] = {};
      bool ok = true;
      for (int u = unit0; ok && u < num_units; u += unit_step) {
        int mt[HALVES], nt;
        unit_coords(u, mt, nt);
        const int n0 = nt * BN_OUT;
        uint32_t bytes = B_BYTES;
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
          if (mt[h] >= 0) bytes += A_BYTES;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, &abort_flag, status, kSiteEmpty)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full_bar[stage]);
          uint8_t* sa = smem + stage * STAGE_BYTES;
          uint8_t* sb = sa + HALVES * A_BYTES;   // the W tile follows the A tiles
          mbar_arrive_expect_tx(fb, bytes);
#pragma unroll
          for (int h = 0; h < HALVES; ++h)
            if (mt[h] >= 0) tma_load_2d(smem_u32(sa + h * A_BYTES), &tmA, fb, kb * BK, mt[h] * BM);
          if constexpr (GEGLU) {
            // gate rows n0.. into the first 128 B-tile rows, up rows N + n0.. after them
            tma_load_2d(smem_u32(sb), &tmB, fb, kb * BK, n0);
            tma_load_2d(smem_u32(sb + B_BYTES / 2), &tmB, fb, kb * BK, N + n0);
          } else if (epi.n1 > 0 && n0 >= epi.n1) {
            tma_load_2d(smem_u32(sb), &tmB2, fb, kb * BK, n0 - epi.n1);
          } else {
            tma_load_2d(smem_u32(sb), &tmB, fb, kb * BK, n0);
          }
          ++fills[stage];
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      // Let every copy this CTA issued land before shared memory is released.
      for (int s = 0; s < STAGES; ++s)
        if (fills[s] > 0) mbar_wait_drain(smem_u32(&full_bar[s]), (fills[s] - 1) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: the whole warp runs the loop (its state
    // warp-uniform); each tcgen05 instruction is issued by one elected lane.
    const uint32_t lead = elect_one();
    const uint32_t idesc_full = idesc_f16(BM, BN, AB_BF16, 0, 0);
    // A plain output's last tile column holding at most half a tile runs
    // MMAs half as wide (the rows of W past N are zeros either way).
    const uint32_t idesc_half = idesc_f16(BM, BN / 2, AB_BF16, 0, 0);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    // the four K=16 MMAs of one 64-deep stage into accumulator d
    auto mma_stage = [&](uint32_t d, uint32_t a_addr, uint32_t b_addr, uint32_t idesc, int kb) {
#pragma unroll
      for (int k = 0; k < BK / 16; ++k)
        mma_ss_lead(lead, d, sdesc_sw128(a_addr + k * 32, 16, 1024),
                    sdesc_sw128(b_addr + k * 32, 16, 1024), idesc, (kb | k) != 0);
    };
    if constexpr (HALVES == 1) {
      int abuf = 0;
      uint32_t aphase = 0;
      for (int u = unit0; ok && u < num_units; u += unit_step) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&acce_bar[abuf]), aphase ^ 1, &abort_flag,
                                               status, kSiteAccEmpty)))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tbase + abuf * BN;
        int mt_u[1], nt_u;
        unit_coords(u, mt_u, nt_u);
        const uint32_t idesc =
            (EPI == kEpiPlain && N - nt_u * BN_OUT <= BN / 2) ? idesc_half : idesc_full;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full_bar[stage]), phase, &abort_flag,
                                                 status, kSiteFull))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
          mma_stage(d_tmem, a_addr, a_addr + A_BYTES, idesc, kb);
          mma_commit_lead(lead, smem_u32(&empty_bar[stage]));
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit_lead(lead, smem_u32(&accf_bar[abuf]));
        abuf ^= 1;
        if (abuf == 0) aphase ^= 1;
      }
    } else {
      // Two halves: half h accumulates at TMEM column h * BN.  A tile's
      // half-0 MMAs start once the epilogue has drained half 0 of the tile
      // before; its half-1 MMAs start once half 1 is drained too.  Until
      // then each stage stays held after its half-0 MMAs (at most all but
      // one, so the producer can still fill the next), and the held stages
      // get their half-1 MMAs, oldest first, as soon as half 1 is free.
      uint32_t tpar = 0;   // parity of this tile's accumulator phases
      for (int u = unit0; ok && u < num_units; u += unit_step) {
        int mt_u[HALVES], nt_u;
        unit_coords(u, mt_u, nt_u);
        const bool two = mt_u[1] >= 0;   // the unit's second half holds rows
        const uint32_t idesc =
            (EPI == kEpiPlain && N - nt_u * BN_OUT <= BN / 2) ? idesc_half : idesc_full;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&acce_bar[0]), tpar ^ 1, &abort_flag,
                                               status, kSiteAccEmpty)))
          break;
        tc_fence_after();
        bool have1 = false;        // half 1's accumulator is free for this tile
        int held = 0, hs0 = 0, hkb0 = 0;   // held stages: count, first slot, its k block
        auto catch_up = [&]() {
          for (int i = 0; i < held; ++i) {
            int s = hs0 + i;
            if (s >= STAGES) s -= STAGES;
            const uint32_t a_addr = smem_u32(smem + s * STAGE_BYTES);
            mma_stage(tbase + BN, a_addr + A_BYTES, a_addr + 2 * A_BYTES, idesc, hkb0 + i);
            mma_commit_lead(lead, smem_u32(&empty_bar[s]));
          }
          held = 0;
        };
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full_bar[stage]), phase, &abort_flag,
                                                 status, kSiteFull))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t b_addr = a_addr + 2 * A_BYTES;
          mma_stage(tbase, a_addr, b_addr, idesc, kb);
          if (two && !have1) {
            if (held + 1 >= STAGES) {
              // every stage would be held: wait for half 1
              if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&acce_bar[1]), tpar ^ 1,
                                                     &abort_flag, status, kSiteAccEmpty))) {
                ok = false;
                break;
              }
              have1 = true;
            } else {
              have1 = __shfl_sync(0xffffffffu,
                                  mbar_test(smem_u32(&acce_bar[1]), tpar ^ 1) ? 1 : 0, 0) != 0;
            }
            if (have1) {
              tc_fence_after();
              catch_up();
            }
          }
          if (!two || have1) {
            if (two) mma_stage(tbase + BN, a_addr + A_BYTES, b_addr, idesc, kb);
            mma_commit_lead(lead, smem_u32(&empty_bar[stage]));
          } else {
            if (held == 0) {
              hs0 = stage;
              hkb0 = kb;
            }
            ++held;
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if (!have1) {
          // half 1 unused by this unit, or not yet free: its phase is
          // waited for every tile, so the two halves' phases stay paired
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&acce_bar[1]), tpar ^ 1, &abort_flag,
                                                 status, kSiteAccEmpty)))
            break;
          tc_fence_after();
          catch_up();
        }
        mma_commit_lead(lead, smem_u32(&accf_bar[0]));
        tpar ^= 1;
      }
    }
    // Drain the tensor pipe before TMEM is released.
    mma_commit_lead(lead, smem_u32(&drain_bar));
    mbar_wait_drain(smem_u32(&drain_bar), 0);
  } else if (warp >= 4) {
    // ---------------- epilogue: TMEM -> registers -> swizzled staging -> TMA store
    const int q = warp - 4;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    uint8_t* staging = smem + STAGES * STAGE_BYTES + q * 2 * STAGING_BYTES;
    int abuf = 0, nchunk = 0;
    uint32_t aphase = 0;
    for (int u = unit0; u < num_units + zero_units; u += unit_step) {
      const bool zero = u >= num_units;   // a pad-only tile: zeros, no accumulator
      int mts[HALVES], nt;
      if (zero) {
        zero_coords(u - num_units, mts[0], nt);
#pragma unroll
        for (int hf = 1; hf < HALVES; ++hf) mts[hf] = -1;
      } else {
        unit_coords(u, mts, nt);
      }
      if (!zero) {
        bool ok = mbar_wait(smem_u32(&accf_bar[abuf]), aphase, &abort_flag, status, kSiteAccFull);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
      }
      const int n0 = nt * BN_OUT;
      const bool seg1 = epi.n1 > 0 && n0 >= epi.n1;     // second output segment
      const int col_off = seg1 ? epi.n1 : 0;              // its first global column
      const CUtensorMap* tcp = seg1 ? &tmC2 : &tmC;
#pragma unroll 1
      for (int half = 0; half < HALVES; ++half) {
        // this half's accumulator: buffer abuf of a one-half tile, or the
        // TMEM columns of half `half` of a two-half tile
        const int ab = HALVES == 2 ? half : abuf;
        if (mts[half] < 0) {
          // a second half past the last M tile: nothing to drain, but its
          // barrier phase stays paired with the first half's
          if (!zero) {
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acce_bar[ab]));
          }
          continue;
        }
        const int mt = mts[half];
        const int m0 = mt * BM;
        const bool rows_in = m0 + q * 32 < M;   // this warp's 32 rows hold some of C
        const uint32_t acc = tbase + lane_off + ab * BN;
        // Stage one 32-row x 128-byte chunk of this warp and store it with TMA
        // (col0 is a global column of C).
        auto stage_store = [&](const uint32_t (&w)[32], int col0) {
          // The staging buffer used two chunks ago must have been read by its store.
          uint8_t* buf = staging + (nchunk & 1) * STAGING_BYTES;
          if (lane == 0 && nchunk >= 2) bulk_wait_group_read<1>();
          __syncwarp();
          // row `lane`, 16-byte unit u lands at unit u ^ (lane % 8) (128-byte swizzle)
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(buf + lane * 128 + ((u ^ (lane & 7)) << 4)) =
                make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (rows_in) tma_store_2d(tcp, smem_u32(buf), col0 - col_off, m0 + q * 32);
            bulk_commit_group();
          }
          ++nchunk;
        };
        auto release_acc = [&]() {
          // last TMEM read of this tile: the accumulator may be reused
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&acce_bar[ab]));
        };
        if (zero) {
          for (int c = 0; c < BN_OUT / CW; ++c) {
            const int col0 = n0 + c * CW;
            if (col0 >= N) break;   // warp-uniform
            uint8_t* buf = staging + (nchunk & 1) * STAGING_BYTES;
            if (lane == 0 && nchunk >= 2) bulk_wait_group_read<1>();
            __syncwarp();
#pragma unroll
            for (int v = 0; v < 8; ++v)
              *reinterpret_cast<uint4*>(buf + lane * 128 + v * 16) = make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (rows_in) tma_store_2d(tcp, smem_u32(buf), col0 - col_off, m0 + q * 32);
              bulk_commit_group();
            }
            ++nchunk;
          }
          continue;
        }
        bool fused = false;
        if constexpr (EPI == kEpiQkNorm)   // warp-uniform
          fused = seg1 ? (n0 - col_off) < epi.n_norm2 : n0 < epi.n_norm;
        if constexpr (EPI == kEpiQkNorm) {
          if (fused) {
            constexpr int HALF = DH / 2;
            constexpr int HEADS = BN / DH;      // head vectors per tile row
            constexpr int PAIRS = HALF / 64;    // 64-column chunk pairs per head
            const int row = m0 + q * 32 + lane;
            const float p = row < M ? static_cast<float>(__ldg(epi.pos + row)) : 0.f;
            const __nv_bfloat16* gam = seg1 ? epi.gamma2 : epi.gamma;
            const float sc_seg = seg1 ? epi.scale2 : epi.scale;
            // d_h = 256 (one head per tile, the short-K 1B shapes where this
            // epilogue is as long as the main loop): the segment's gamma spread
            // over the warp, word k of lane l holding the bf16 pair (gamma_j,
            // gamma_{j + d_h/2}) of j = 32 k + l, fetched with one shuffle per
            // rotated pair (shuffles and loads share the shared-memory data
            // path that feeds the tensor core).  d_h = 128 reads gamma from
            // global memory per use (the shuffles' registers would spill there).
            constexpr bool G_SHFL = DH == 256;
            uint32_t gl[G_SHFL ? HALF / 32 : 1];
#pragma unroll
            for (int k = 0; G_SHFL && k < HALF / 32; ++k) {
              const uint16_t* gb = reinterpret_cast<const uint16_t*>(gam);
              gl[k] = static_cast<uint32_t>(__ldg(gb + k * 32 + lane)) |
                      (static_cast<uint32_t>(__ldg(gb + HALF + k * 32 + lane)) << 16);
            }
            float rs[HEADS];   // 1 / rms of each head, times the segment's scale
#pragma unroll
            for (int e = 0; e < HEADS; ++e) {
              // sum of squares in packed fp32x2 (four partial sums)
              float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
#pragma unroll
              for (int k = 0; k < DH / 64; ++k) {
                uint32_t a0[32], a1[32];
                tmem_ld32(acc + e * DH + k * 64, a0);
                tmem_ld32(acc + e * DH + k * 64 + 32, a1);
                tmem_ld_wait(a0);
                tmem_ld_wait(a1);
#pragma unroll
                for (int t = 0; t < 32; t += 2) {
                  const float2 u = make_float2(__uint_as_float(a0[t]), __uint_as_float(a0[t + 1]));
                  const float2 w = make_float2(__uint_as_float(a1[t]), __uint_as_float(a1[t + 1]));
                  sa = __ffma2_rn(u, u, sa);
                  sb = __ffma2_rn(w, w, sb);
                }
              }
              const float ss = (sa.x + sa.y) + (sb.x + sb.y);
              rs[e] = rsqrtf(ss * (1.f / DH) + 1e-6f) * sc_seg;
            }
            // Each pair of 64-column chunks (first half, partner half) goes to
            // the two staging buffers: the first-half chunk to buffer 0, the
            // partner chunk to buffer 1 (nchunk is even here).
            uint8_t* buf_a = staging;
            uint8_t* buf_b = staging + STAGING_BYTES;
            // Blocks of 32 rotated pairs (head e, chunk pair i, 32-column half
            // h): a runtime loop over the blocks, each block unrolled.  Fully
            // unrolled, this epilogue is tens of KB of instructions, and
            // streaming through them every tile evicts the MMA issuer's and the
            // TMA producer's loops from the instruction caches they share.
            constexpr int N_BLK = HEADS * PAIRS * 2;
#pragma unroll 1
            for (int blk = 0; blk < N_BLK; ++blk) {
              const int e = blk / (2 * PAIRS), i = (blk >> 1) % PAIRS, h = blk & 1;
              const int ca = e * (DH / 64) + i, cb = ca + PAIRS;   // first-half, partner chunk
              const int jb = i * 64 + h * 32;                     // first pair index of the block
              float rse = rs[0];
#pragma unroll
              for (int k = 1; k < HEADS; ++k)
                if (e == k) rse = rs[k];
              uint32_t gw = 0;   // this block's gamma word of each lane
              if constexpr (G_SHFL) {
#pragma unroll
                for (int k = 0; k < HALF / 32; ++k)
                  if ((jb >> 5) == k) gw = gl[k];
              }
              const float2* fr = epi.freqs.f + jb;
              uint32_t x1[32], x2[32];
              tmem_ld32(acc + ca * 64 + h * 32, x1);
              tmem_ld32(acc + cb * 64 + h * 32, x2);
              tmem_ld_wait(x1);
              tmem_ld_wait(x2);
              if (blk == N_BLK - 1) release_acc();
              uint32_t wa[16], wb[16];
              const float2 rs2 = make_float2(rse, rse), nrs2 = make_float2(-rse, -rse);
              // Two rotated pairs (j, j + 1), j = jb + t, per step in packed
              // fp32x2 arithmetic.
#pragma unroll
              for (int t = 0; t < 32; t += 2) {
                float2 g1, g2;   // (gamma_j, gamma_{j+1}), their partners at j + d_h/2
                if constexpr (G_SHFL) {
                  const uint32_t ga = __shfl_sync(0xffffffffu, gw, t);
                  const uint32_t gb = __shfl_sync(0xffffffffu, gw, t + 1);
                  g1 = make_float2(__uint_as_float(ga << 16), __uint_as_float(gb << 16));
                  g2 = make_float2(__uint_as_float(ga & 0xffff0000u),
                                   __uint_as_float(gb & 0xffff0000u));
                } else {
                  g1 = make_float2(__bfloat162float(gam[jb + t]), __bfloat162float(gam[jb + t + 1]));
                  g2 = make_float2(__bfloat162float(gam[jb + t + HALF]),
                                   __bfloat162float(gam[jb + t + 1 + HALF]));
                }
                const float2 xa = make_float2(__uint_as_float(x1[t]), __uint_as_float(x1[t + 1]));
                const float2 xb = make_float2(__uint_as_float(x2[t]), __uint_as_float(x2[t + 1]));
                // x (1 + gamma) as one fused multiply-add per lane
                const float2 y1 = __ffma2_rn(xa, g1, xa);
                const float2 y2 = __ffma2_rn(xb, g2, xb);
                float2 sn, cs;
                rope_sincos2(p, fr[t], fr[t + 1], sn, cs);
                // (y1 cos - y2 sin) / rms and (y2 cos + y1 sin) / rms, the
                // scale taken into cos and sin
                const float2 c = __fmul2_rn(cs, rs2), s = __fmul2_rn(sn, rs2);
                const float2 ns = __fmul2_rn(sn, nrs2);
                const float2 o1 = __ffma2_rn(y1, c, __fmul2_rn(y2, ns));
                const float2 o2 = __ffma2_rn(y2, c, __fmul2_rn(y1, s));
                wa[t / 2] = pack_half2(o1.x, o1.y);
                wb[t / 2] = pack_half2(o2.x, o2.y);
              }
              if (h == 0) {
                // both buffers must have been read by the earlier stores
                if (lane == 0 && nchunk > 0) bulk_wait_group_read<0>();
                __syncwarp();
              }
              // row `lane`, 16-byte unit u at unit u ^ (lane % 8) (128-byte swizzle)
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int pu = ((4 * h + u) ^ (lane & 7)) << 4;
                *reinterpret_cast<uint4*>(buf_a + lane * 128 + pu) =
                    make_uint4(wa[4 * u], wa[4 * u + 1], wa[4 * u + 2], wa[4 * u + 3]);
                *reinterpret_cast<uint4*>(buf_b + lane * 128 + pu) =
                    make_uint4(wb[4 * u], wb[4 * u + 1], wb[4 * u + 2], wb[4 * u + 3]);
              }
              if (h == 1) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  // one bulk group per buffer: a plain chunk that follows waits
                  // for all but the newest group, i.e. for buffer 0's store
                  if (rows_in) tma_store_2d(tcp, smem_u32(buf_a), n0 - col_off + ca * 64, m0 + q * 32);
                  bulk_commit_group();
                  if (rows_in) tma_store_2d(tcp, smem_u32(buf_b), n0 - col_off + cb * 64, m0 + q * 32);
                  bulk_commit_group();
                }
                nchunk += 2;
              }
            }
          }
        }
        for (int c = 0; !fused && c < BN_OUT / CW; ++c) {
          const int col0 = n0 + c * CW;
          if (col0 >= N) break;   // warp-uniform
          // 128 bytes of this thread's row: 8 x 16-byte units
          uint32_t w[32];
          if constexpr (sizeof(OutT) == 4) {
            tmem_ld32(acc + c * 32, w);
            tmem_ld_wait(w);
          } else {
            uint32_t r0[32], r1[32];
            tmem_ld32(acc + c * 64, r0);
            tmem_ld32(acc + c * 64 + 32, r1);
            if constexpr (GEGLU) {
              uint32_t u0[32], u1[32];
              tmem_ld32(acc + BN / 2 + c * 64, u0);
              tmem_ld32(acc + BN / 2 + c * 64 + 32, u1);
              tmem_ld_wait(r0);
              tmem_ld_wait(r1);
              tmem_ld_wait(u0);
              tmem_ld_wait(u1);
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                w[e] = pack2<OutT>(gelu_tanh_mul(__uint_as_float(r0[2 * e]), __uint_as_float(u0[2 * e])),
                                   gelu_tanh_mul(__uint_as_float(r0[2 * e + 1]),
                                                 __uint_as_float(u0[2 * e + 1])));
                w[16 + e] =
                    pack2<OutT>(gelu_tanh_mul(__uint_as_float(r1[2 * e]), __uint_as_float(u1[2 * e])),
                                gelu_tanh_mul(__uint_as_float(r1[2 * e + 1]),
                                              __uint_as_float(u1[2 * e + 1])));
              }
            } else {
              tmem_ld_wait(r0);
              tmem_ld_wait(r1);
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                w[e] = pack2<OutT>(__uint_as_float(r0[2 * e]), __uint_as_float(r0[2 * e + 1]));
                w[16 + e] = pack2<OutT>(__uint_as_float(r1[2 * e]), __uint_as_float(r1[2 * e + 1]));
              }
            }
          }
          if (c == BN_OUT / CW - 1 || col0 + CW >= N) release_acc();
          stage_store(w, col0);
        }
      }
      if (!zero) {
        if (HALVES == 1) {
          abuf ^= 1;
          if (abuf == 0) aphase ^= 1;
        } else {
          aphase ^= 1;
        }
      }
    }
    if (lane == 0) bulk_wait_group_all();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

// Rows per tile: 0 chooses (see launch_typed), 128 or 256 forces one.
std::atomic<int> g_tile_rows{0};

// The launch of one instantiation: grid (one CTA per SM, at most one per
// unit) and the L2 grouping of M tiles (in units of HALVES 128-row tiles).
template <int AB_BF16, typename OutT, int EPI, int DH, int HALVES>
cudaError_t launch_kernel(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                          const CUtensorMap& tb2, const CUtensorMap& tc2, int M, int N, int K,
                          cudaStream_t stream, int* status, int max_ctas, const QkEpi& epi,
                          const int32_t* pad_lens, int seg_T, int zero_from) {
  constexpr bool GEGLU = EPI == kEpiGeglu;
  constexpr uint32_t smem_bytes = Ring<HALVES>::SMEM_BYTES;
  auto kern = pad_lens != nullptr ? gemm_tn_kernel<AB_BF16, OutT, EPI, DH, true, HALVES>
                                  : gemm_tn_kernel<AB_BF16, OutT, EPI, DH, false, HALVES>;
  if (cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), smem_bytes)) return e;
  const int bn_out = GEGLU ? BN / 2 : BN;
  const int m_tiles = (M + BM - 1) / BM;
  const int mu_units = (m_tiles + HALVES - 1) / HALVES;
  const int units = mu_units * ((N + bn_out - 1) / bn_out);
  int grid = num_sms();
  if (max_ctas > 0 && max_ctas < grid) grid = max_ctas;
  if (units < grid) grid = units;
  const size_t a_tile_bytes = static_cast<size_t>(BM) * K * 2;
  const size_t w_bytes = static_cast<size_t>(GEGLU ? 2 * N : N) * K * 2;
  int group_m = kSmallGroupM;
  if (w_bytes > kSmallWeightBytes) {
    const size_t g = kGroupBytes / a_tile_bytes;
    if (g > static_cast<size_t>(group_m)) group_m = static_cast<int>(g);
  }
  group_m = group_m / HALVES > 1 ? group_m / HALVES : 1;
  if (group_m > mu_units) group_m = mu_units;
  return launch_pdl(kern, dim3(grid), dim3(THREADS), smem_bytes, stream, ta, tb, tc, tb2, tc2, M,
                    N, K, group_m, pad_lens, seg_T, zero_from, status, epi);
}

// C (and, for a split launch, the second segment's C2 with ldc2 and the
// second weight map tb2; epi.n1 > 0) as 32-row x 128-byte TMA tiles.
// Plain outputs with K of 512 or more, and GeGLU outputs with K of 2048 or
// more, take two-half (256-row) tiles unless the last wave of their units
// would run too empty.  The epilogue of a two-half tile is not hidden behind
// a main loop, so a short K pays it more often, and GeGLU's is the longer
// (measured: 256-row GeGLU +2.5% at K = 2560, -3.5% at K = 1152).  The fused
// prologue, whose epilogue is as long as a short main loop, keeps one-half
// tiles.
template <int AB_BF16, typename OutT, int EPI = kEpiPlain, int DH = 0>
cudaError_t launch_typed(const CUtensorMap& ta, const CUtensorMap& tb, void* C, long ldc, int M,
                         int N, int K, cudaStream_t stream, int* status, int max_ctas,
                         const QkEpi& epi = QkEpi{}, const CUtensorMap* tb2 = nullptr,
                         void* C2 = nullptr, long ldc2 = 0, const int32_t* pad_lens = nullptr,
                         int seg_T = 0, int zero_from = 0) {
  // Output tile map: boxes of 32 rows x 128 bytes, 128-byte swizzle.
  CUtensorMap tc;
  const CUtensorMapDataType cdt = sizeof(OutT) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                  : std::is_same<OutT, __half>::value
                                      ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t n_seg0 = epi.n1 > 0 ? static_cast<uint64_t>(epi.n1) : static_cast<uint64_t>(N);
  const uint64_t cdims[2] = {n_seg0, static_cast<uint64_t>(M)};
  const uint64_t cstr[1] = {static_cast<uint64_t>(ldc) * sizeof(OutT)};
  const uint32_t cbox[2] = {static_cast<uint32_t>(128 / sizeof(OutT)), 32};
  if (!encode_tiled(&tc, cdt, 2, C, cdims, cstr, cbox)) return cudaErrorInvalidValue;
  CUtensorMap tc2 = tc;
  if (epi.n1 > 0) {
    const uint64_t cdims2[2] = {static_cast<uint64_t>(N - epi.n1), static_cast<uint64_t>(M)};
    const uint64_t cstr2[1] = {static_cast<uint64_t>(ldc2) * sizeof(OutT)};
    if (tb2 == nullptr || C2 == nullptr || !encode_tiled(&tc2, cdt, 2, C2, cdims2, cstr2, cbox))
      return cudaErrorInvalidValue;
  }
  const CUtensorMap& tbb = tb2 != nullptr ? *tb2 : tb;
  if constexpr (EPI != kEpiQkNorm) {
    const int rows = g_tile_rows.load(std::memory_order_relaxed);
    bool two = rows == 256;
    if (rows == 0 && K >= (EPI == kEpiGeglu ? 2048 : 512)) {
      // A two-half tile does the work of two one-half tiles in ~1/1.12 of
      // their time (measured, K = 1024-10240); it pays where its waves of
      // units over the grid do not outnumber that.
      const int bn_out = EPI == kEpiGeglu ? BN / 2 : BN;
      const int n_tiles = (N + bn_out - 1) / bn_out, m_tiles = (M + BM - 1) / BM;
      int grid = num_sms();
      if (max_ctas > 0 && max_ctas < grid) grid = max_ctas;
      const long waves1 = (static_cast<long>(m_tiles) * n_tiles + grid - 1) / grid;
      const long waves2 = (static_cast<long>((m_tiles + 1) / 2) * n_tiles + grid - 1) / grid;
      two = waves2 * 200 <= waves1 * 112;
    }
    if (two)
      return launch_kernel<AB_BF16, OutT, EPI, DH, 2>(ta, tb, tc, tbb, tc2, M, N, K, stream,
                                                      status, max_ctas, epi, pad_lens, seg_T,
                                                      zero_from);
  }
  return launch_kernel<AB_BF16, OutT, EPI, DH, 1>(ta, tb, tc, tbb, tc2, M, N, K, stream, status,
                                                  max_ctas, epi, pad_lens, seg_T, zero_from);
}

bool encode_ab(CUtensorMap& ta, CUtensorMap& tb, const void* A, long lda, const void* W, long ldw,
               int M, int N_rows, int K, int in_dtype, uint32_t b_box_rows) {
  const CUtensorMapDataType tdt =
      in_dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t adims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
  const uint64_t astr[1] = {static_cast<uint64_t>(lda) * 2};
  const uint32_t abox[2] = {BK, BM};
  const uint64_t bdims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N_rows)};
  const uint64_t bstr[1] = {static_cast<uint64_t>(ldw) * 2};
  const uint32_t bbox[2] = {BK, b_box_rows};
  return encode_tiled(&ta, tdt, 2, A, adims, astr, abox) &&
         encode_tiled(&tb, tdt, 2, W, bdims, bstr, bbox);
}

}  // namespace

int set_gemm_tile_rows(int rows) {
  if (rows != 0 && rows != 128 && rows != 256) return -1;
  return g_tile_rows.exchange(rows);
}

cudaError_t launch_linear(const void* A, long lda, const void* W, long ldw, void* C, long ldc,
                          int M, int N, int K, int in_dtype, int out_dtype, cudaStream_t stream,
                          int* status, int max_ctas, const int32_t* pad_lens, int seg_T,
                          bool zero_pad_tiles) {
  if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
  if (in_dtype != kBF16 && in_dtype != kF16) return cudaErrorInvalidValue;
  if (M <= kSkinnyMaxRows)
    return launch_linear_skinny(A, lda, W, ldw, C, ldc, M, N, K, in_dtype, out_dtype, stream,
                                status);
  CUtensorMap ta, tb;
  if (!encode_ab(ta, tb, A, lda, W, ldw, M, N, K, in_dtype, BN)) return cudaErrorInvalidValue;
  const int zf = zero_pad_tiles ? 0 : N;   // zeros in every column of pad-only tiles, or none
#define G3_GEMM_OUT(AB)                                                                        \
  switch (out_dtype) {                                                                         \
    case kF32:                                                                                 \
      return launch_typed<AB, float>(ta, tb, C, ldc, M, N, K, stream, status, max_ctas, {},    \
                                     nullptr, nullptr, 0, pad_lens, seg_T, zf);                \
    case kF16:                                                                                 \
      return launch_typed<AB, __half>(ta, tb, C, ldc, M, N, K, stream, status, max_ctas, {},   \
                                      nullptr, nullptr, 0, pad_lens, seg_T, zf);               \
    case kBF16:                                                                                \
      return launch_typed<AB, __nv_bfloat16>(ta, tb, C, ldc, M, N, K, stream, status,       \
                                             max_ctas, {}, nullptr, nullptr, 0, pad_lens,      \
                                             seg_T, zf);                                       \
    default: return cudaErrorInvalidValue;                                                     \
  }
  if (in_dtype == kBF16) {
    G3_GEMM_OUT(1)
  }
  G3_GEMM_OUT(0)
#undef G3_GEMM_OUT
}

cudaError_t launch_geglu(const void* A, long lda, const void* Wgu, long ldw, void* Z, long ldz,
                         int M, int D_ff, int K, int in_dtype, cudaStream_t stream, int* status) {
  if (M <= 0 || D_ff <= 0 || K <= 0) return cudaSuccess;
  if (in_dtype != kBF16 && in_dtype != kF16) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!encode_ab(ta, tb, A, lda, Wgu, ldw, M, 2 * D_ff, K, in_dtype, BN / 2))
    return cudaErrorInvalidValue;
  if (in_dtype == kBF16)
    return launch_typed<1, __half, kEpiGeglu>(ta, tb, Z, ldz, M, D_ff, K, stream, status, 0);
  return launch_typed<0, __half, kEpiGeglu>(ta, tb, Z, ldz, M, D_ff, K, stream, status, 0);
}

bool linear_qknorm_fusable(int M, int N, int n_norm, int d_h) {
  return M > kSkinnyMaxRows && (d_h == 128 || d_h == 256) && n_norm > 0 && n_norm <= N &&
         n_norm % BN == 0;
}

cudaError_t launch_qkv_qknorm(const void* A, long lda, const void* Wq, const void* Wkv, long ldw,
                              void* Qout, long ldq, void* KVout, long ldkv, int M, int HD, int KVD,
                              int K, int in_dtype, const void* gamma_q, const void* gamma_k,
                              const int32_t* pos, int d_h, double rope_base, double rope_scale,
                              float query_scale, cudaStream_t stream, int* status,
                              const int32_t* pad_lens, int seg_T) {
  if (M <= 0 || K <= 0) return cudaSuccess;
  if (in_dtype != kBF16 && in_dtype != kF16) return cudaErrorInvalidValue;
  if (!linear_qknorm_fusable(M, HD, HD, d_h) || !linear_qknorm_fusable(M, 2 * KVD, KVD, d_h))
    return cudaErrorInvalidValue;
  CUtensorMap ta, tb, ta2, tb2;
  if (!encode_ab(ta, tb, A, lda, Wq, ldw, M, HD, K, in_dtype, BN) ||
      !encode_ab(ta2, tb2, A, lda, Wkv, ldw, M, 2 * KVD, K, in_dtype, BN))
    return cudaErrorInvalidValue;
  QkEpi epi{};
  epi.freqs = make_rope_freqs(d_h, rope_base, rope_scale);
  epi.gamma = static_cast<const __nv_bfloat16*>(gamma_q);
  epi.gamma2 = static_cast<const __nv_bfloat16*>(gamma_k);
  epi.pos = pos;
  epi.n_norm = HD;
  epi.n_norm2 = KVD;
  epi.n1 = HD;
  epi.scale = query_scale;
  epi.scale2 = 1.f;
  const int N = HD + 2 * KVD;
#define G3_QKV(AB, DH_)                                                                        \
  return launch_typed<AB, __half, kEpiQkNorm, DH_>(ta, tb, Qout, ldq, M, N, K, stream, status, 0, \
                                                   epi, &tb2, KVout, ldkv, pad_lens, seg_T,    \
                                                   HD + KVD);
  if (in_dtype == kBF16) {
    if (d_h == 256) G3_QKV(1, 256)
    G3_QKV(1, 128)
  }
  if (d_h == 256) G3_QKV(0, 256)
  G3_QKV(0, 128)
#undef G3_QKV
}

cudaError_t launch_linear_qknorm(const void* A, long lda, const void* W, long ldw, void* C,
                                 long ldc, int M, int N, int K, int in_dtype, const void* gamma,
                                 const int32_t* pos, int d_h, int n_norm, double rope_base,
                                 double rope_scale, float scale, cudaStream_t stream,
                                 int* status) {
  if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
  if (in_dtype != kBF16 && in_dtype != kF16) return cudaErrorInvalidValue;
  if (!linear_qknorm_fusable(M, N, n_norm, d_h)) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!encode_ab(ta, tb, A, lda, W, ldw, M, N, K, in_dtype, BN)) return cudaErrorInvalidValue;
  QkEpi epi{};
  epi.freqs = make_rope_freqs(d_h, rope_base, rope_scale);
  epi.gamma = static_cast<const __nv_bfloat16*>(gamma);
  epi.pos = pos;
  epi.n_norm = n_norm;
  epi.scale = scale;
#define G3_QKN(AB, DH_)                                                                      \
  return launch_typed<AB, __half, kEpiQkNorm, DH_>(ta, tb, C, ldc, M, N, K, stream, status, 0, \
                                                   epi);
  if (in_dtype == kBF16) {
    if (d_h == 256) G3_QKN(1, 256)
    G3_QKN(1, 128)
  }
  if (d_h == 256) G3_QKN(0, 256)
  G3_QKN(0, 128)
#undef G3_QKN
}

}  // namespace g3
