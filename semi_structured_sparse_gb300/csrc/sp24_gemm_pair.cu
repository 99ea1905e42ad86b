// sp24_gemm_pair.cu -- the 2:4 sparse e4m3 GEMM on SM pairs (tcgen05
// cta_group::2), for large token counts with per-token x per-channel scaling
// (the per-tensor-K case of the group-wise scheme: gK = K).
//
// Why pairs.  With one CTA per 128-row weight tile and 256 tokens, each
// 128-wide K block brings 8 KB of kept values, 2 KB of metadata and 32 KB of
// activations into one SM for 320 cycles of tensor work.  A pair of SMs
// issues M = 256 MMAs instead: each SM holds its own 128 weight rows and only
// half of the 256 activation rows (the tensor cores exchange B across the
// pair), so a K block is 26 KB per SM for the same 320 cycles.
//
// Math and layout are those of the one-CTA kernel (sp24_gemm.cu): Y^T = W X^T
// with the sparse weight as the A operand, a weight row per TMEM lane, a token
// per TMEM column, and Y[m][n] = bf16(sx[m] sw[n] sum_k Wq[n][k] Xq[m][k]).
//
// Pipeline.  A stage holds KS = 2 consecutive K blocks (52 KB per SM): each
// mbarrier round trip between loads and MMAs costs a few hundred cycles of
// latency whatever the stage size, and four 52 KB stages keep more bytes in
// flight than seven 26 KB ones.
//
// Roles (both CTAs of a pair run the same warps; the even CTA is the leader):
//   warps 0-1  producers, alternating stages: each CTA loads its weight tiles
//              (values, metadata) and its half of the activation tiles with
//              TMA; all copies signal the LEADER's full barrier, which the
//              leader's producer arms with both CTAs' bytes.
//   warp 2     TMEM allocation (pair-collective).  In the leader one lane
//              issues, per K block, tcgen05.cp of the metadata (each CTA into
//              its own TMEM) and two sparse M = 256 MMAs; per stage it commits
//              to both CTAs' empty barriers and, after a tile, to both
//              accumulator-full barriers.
//   warps 3-10 epilogue, in each CTA: drain its 128 x 256 accumulator into
//              registers, release it to the leader, scale, convert to bf16
//              and TMA-store its 128 channels.  While the next tile runs, the
//              conversion goes through a 64-token staging buffer in four
//              passes; for the CTA's last tile the idle stage ring holds the
//              whole tile and the stores go out at once.
//
// Fused side GEMM (SIDE, CUTLASS issue #2058: Y = X1 W1^T + X2 W2^T in one
// kernel).  Token tiles are then 240 wide, so that TMEM holds the main
// accumulator (columns 0-239), the side accumulator (240-479) and an 8-slot
// metadata ring (480-511, one slot per K block in flight).  Each tile starts
// with one extra pipeline stage that carries the W2 tile of the CTA's 128
// channels and the X2 rows of its 120 tokens (bf16, 128-byte swizzle); the
// MMA thread turns it into r / 16 bf16 M = 256 MMAs into the side
// accumulator.  The epilogue forms bf16((sx sw) acc + side).
//
// The kernel is launched with programmatic stream serialisation: its
// prologue (barriers, TMEM, descriptor prefetch) overlaps the previous
// kernel's tail, and pdl_wait() precedes every global-memory access.
#include <cuda_bf16.h>
#include <atomic>
#include "sp24_gemm_common.cuh"

namespace sp24 {
namespace {

constexpr int KS = 2;                          // K blocks per stage
constexpr int VROWS = A_STAGE / 128;           // a values tile is 64 rows of 128 B
constexpr int MROWS = META_STAGE / 128;        // a metadata tile is 16 rows of 128 B
constexpr int SIDE_COL = 240;                  // first TMEM column of the side accumulator
constexpr int SIDE_W2_BYTES = BM * 128;        // side stage: W2 tile (128 channels x 64 bf16)

template <int PN_, bool SIDE_, bool PROMOTE_ = false>
struct PairCfg {
  static constexpr int PN = PN_;                    // tokens per pair tile (MMA N)
  static constexpr bool SIDE = SIDE_;
  static constexpr bool PROMOTE = PROMOTE_;         // group-wise scales: one partial per K block
  static constexpr int HALF_N = PN / 2;             // activation rows each CTA loads
  static constexpr int P_B = HALF_N * BK;           // activations per CTA per K block
  static constexpr int A_OFF = 0;                   // KS values tiles (contiguous in the tiled storage)
  static constexpr int META_OFF = KS * A_STAGE;     // KS metadata tiles
  static constexpr int B_OFF = KS * (A_STAGE + META_STAGE);
  static constexpr int LOAD_BYTES = B_OFF + KS * P_B;  // TMA bytes each CTA receives per stage
  // promotion: per K block of the stage a 1 KB scale slot, sx of the pair
  // tile's PN tokens then sw of this CTA's 128 channels (cp.async)
  static constexpr int SCL_OFF = LOAD_BYTES;
  static constexpr int STAGE = LOAD_BYTES + (PROMOTE ? KS * 1024 : 0);
  // TMEM accumulators of PN columns: promotion keeps one partial per K block in
  // flight in each, three of 128 tokens or four of 112 beside the metadata ring
  static constexpr int NACC = PROMOTE ? (PN <= 112 ? 4 : 3) : 1;
  // token chunk (warp half h holds chunks h, h + 2, ...): 32, or 24 when a
  // warp's PN / 2 tokens are not a multiple of 32 (240-token tiles); under
  // promotion with 112-token tiles, the warp's 56 tokens in one chunk
  static constexpr int CHUNK = (PN / 2) % 32 == 0 ? 32 : (PROMOTE ? PN / 2 : 24);
  // tokens per staged store pass (promotion stages the whole tile at once)
  static constexpr int OUT_TOKENS = PROMOTE ? PN : 2 * CHUNK;
  static constexpr int OUT_BYTES = OUT_TOKENS * BM * 2;
  static constexpr int SCALE_BYTES = 4 * 256;
  static constexpr int FIXED = 1024 + OUT_BYTES + SCALE_BYTES + BAR_BYTES;
  static constexpr int META_RING = SIDE ? 8 : META_SLOTS;  // metadata slots (4 TMEM columns each)
  static constexpr int META_BASE = SIDE ? 480 : META_COL0;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - FIXED) / STAGE;
  static constexpr int STAGES = STAGES_FIT < META_RING / KS ? STAGES_FIT : META_RING / KS;
  static constexpr int SMEM = FIXED + STAGES * STAGE;
  static constexpr int COLS = PN / 2;               // accumulator columns per epilogue warp
  static constexpr int NCHUNK = COLS / CHUNK;       // chunks per epilogue warp
  static constexpr int NPASS = PN / OUT_TOKENS;
  static constexpr int SIDE_X2_BYTES = HALF_N * 128;  // side stage: this CTA's X2 rows
  static_assert(B_OFF % 1024 == 0 && STAGE % 1024 == 0 && P_B % 1024 == 0, "1024-byte swizzle alignment");
  static_assert(STAGES >= 3 && STAGES <= MAX_STAGES, "pipeline depth");
  static_assert(SIDE ? (PN <= SIDE_COL && SIDE_COL + PN <= META_BASE) : NACC * PN <= META_COL0, "TMEM columns");
  static_assert(!PROMOTE || (!SIDE && PN + BM <= 256), "a scale slot holds PN + 128 floats");
  static_assert(NACC <= 4, "four accumulator barriers");
  static_assert(SCL_OFF % 16 == 0, "scale slots start on a 16-byte boundary (read as float4)");
  static_assert(NCHUNK * CHUNK == COLS && CHUNK % 8 == 0 && OUT_TOKENS * NPASS == PN, "epilogue chunks");
  static_assert(STAGES * STAGE >= PN * BM * 2, "the ring holds a whole output tile");
  static_assert(!SIDE || SIDE_W2_BYTES + SIDE_X2_BYTES <= STAGE, "the side operands fit one stage");
};

// bf16((s_t sw) acc_t [+ add_t] + bias) of 4 consecutive tokens, as two packed words.
template <bool ADD>
__device__ __forceinline__ uint2 scale4_pack(const float* s, float sw, const uint32_t* acc, const uint32_t* add,
                                             float bias) {
  const float4 s4 = *reinterpret_cast<const float4*>(s);
  const float2 b2 = make_float2(bias, bias);
  const float2 a01 = ADD ? __fadd2_rn(make_float2(__uint_as_float(add[0]), __uint_as_float(add[1])), b2) : b2;
  const float2 a23 = ADD ? __fadd2_rn(make_float2(__uint_as_float(add[2]), __uint_as_float(add[3])), b2) : b2;
  const float2 w2 = make_float2(sw, sw);
  const float2 y01 = __ffma2_rn(__fmul2_rn(make_float2(s4.x, s4.y), w2),
                                make_float2(__uint_as_float(acc[0]), __uint_as_float(acc[1])), a01);
  const float2 y23 = __ffma2_rn(__fmul2_rn(make_float2(s4.z, s4.w), w2),
                                make_float2(__uint_as_float(acc[2]), __uint_as_float(acc[3])), a23);
  return make_uint2(bf16x2_rn(y01.x, y01.y), bf16x2_rn(y23.x, y23.y));
}

// Loads N consecutive accumulator columns (N a multiple of 8) of this warp's lanes.
template <int N>
__device__ __forceinline__ void tmem_load_n(uint32_t taddr, uint32_t* r) {
#pragma unroll
  for (int i = 0; i + 16 <= N; i += 16) tmem_ld16(taddr + i, *reinterpret_cast<uint32_t(*)[16]>(r + i));
  if constexpr (N % 16 != 0) tmem_ld8(taddr + (N / 16) * 16, r + (N / 16) * 16);
}

template <int PN, bool SIDE, bool PROMOTE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    sp24_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_m, const __grid_constant__ CUtensorMap tm_y,
                          const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_x2,
                          const GemmArgs p) {
  using C = PairCfg<PN, SIDE, PROMOTE>;
  constexpr int HALF_N = C::HALF_N, CHUNK = C::CHUNK, NACC = C::NACC;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base by pointer arithmetic on the shared array, so that
  // accesses through it compile to shared-memory instructions
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = sm;
  uint8_t* out_tile = sm + C::STAGES * C::STAGE;                   // [2 channel halves][OUT_TOKENS][64] bf16
  float* scl = reinterpret_cast<float*>(out_tile + C::OUT_BYTES);  // token scales of the tile [PN]
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_tile + C::OUT_BYTES + C::SCALE_BYTES);
  uint64_t* full = bars;                  // [STAGES] leader: both CTAs' loads -> MMA
  uint64_t* empty = bars + MAX_STAGES;    // [STAGES] each CTA: MMA done with the stage -> its loads
  uint64_t* accf = bars + 2 * MAX_STAGES; // [NACC] each CTA: accumulator complete -> its epilogue
  uint64_t* acce = accf + 4;              // [NACC] leader: both epilogues drained the accumulator -> MMA
  uint64_t* sfull = acce + 4;             // [STAGES] promotion, each CTA: the stage's scales landed
  uint64_t* drain = sfull + MAX_STAGES;   // leader: every MMA finished (before TMEM is freed)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(num_clusters_x());
  const int num_units = p.m_tiles * p.n_tiles;
  const int k_stages = (p.k_tiles + KS - 1) / KS;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full[i], 1);
      // promotion: the epilogue warps also read the stage (its scales)
      mbar_init(&empty[i], 1 + (PROMOTE ? EPI_WARPS : 0));
      if (PROMOTE) mbar_init(&sfull[i], 32);  // one cp.async arrival per producer lane
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], 2 * EPI_WARPS);  // one arrival per epilogue warp of each CTA
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == MMA_WARP + 1 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_m);
    tma_prefetch_desc(&tm_y);
    if (SIDE) {
      tma_prefetch_desc(&tm_w2);
      tma_prefetch_desc(&tm_x2);
    }
  }
  if (warp == MMA_WARP) {
    tmem_alloc_pair(tslot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers exist and TMEM is allocated before anyone signals across
  tc_fence_after();
  const uint32_t tbase = *tslot;
  pdl_wait();      // the previous kernel's writes are visible from here on

  if (warp < PRODUCERS) {
    // ----------------------------------------------------------- producers
    const uint32_t full0 = cluster_addr(&full[0], 0);  // the leader's full barriers
    int64_t flat = 0;
    bool ok = true;
    for (int u = pair; u < num_units && ok; u += npairs) {
      const int n_tile = 2 * (u % p.n_tiles) + static_cast<int>(rank);  // this CTA's 128 weight rows
      const int m0 = (u / p.n_tiles) * PN + static_cast<int>(rank) * HALF_N;  // this CTA's token rows
      const int vrow = n_tile * p.k_tiles * VROWS;
      const int mrow = n_tile * p.k_tiles * MROWS;
      // with SIDE, stage -1 of the tile carries the side operands
      for (int ks = SIDE ? -1 : 0; ks < k_stages; ++ks, ++flat) {
        if (flat % PRODUCERS != warp) continue;
        const uint32_t stage = static_cast<uint32_t>(flat % C::STAGES);
        const uint32_t phase = static_cast<uint32_t>((flat / C::STAGES) & 1);
        const bool got = mbar_wait<true>(&empty[stage], phase ^ 1);
        if (!__all_sync(0xFFFFFFFFu, got)) { ok = false; break; }
        if (lane == 0) {
          const uint32_t fb = full0 + 8u * stage;
          uint8_t* st = ring + stage * C::STAGE;
          if (SIDE && ks < 0) {
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (SIDE_W2_BYTES + C::SIDE_X2_BYTES));
            tma_load_2d_pair(st, &tm_w2, fb, 0, n_tile * BM);
            tma_load_2d_pair(st + SIDE_W2_BYTES, &tm_x2, fb, 0, m0);
          } else {
            // Always KS blocks: with an odd block count the last stage's second
            // block reads the next weight tile's rows (or zero fill past the end)
            // and K coordinates past K (zero fill); the MMA skips it.
            const int kt = ks * KS;
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * C::LOAD_BYTES);  // both CTAs' bytes
            tma_load_2d_pair(st + C::A_OFF, &tm_v, fb, 0, vrow + kt * VROWS);
            tma_load_2d_pair(st + C::META_OFF, &tm_m, fb, 0, mrow + kt * MROWS);
#pragma unroll
            for (int j = 0; j < KS; ++j) tma_load_2d_pair(st + C::B_OFF + j * C::P_B, &tm_x, fb, (kt + j) * BK, m0);
          }
        }
        if constexpr (PROMOTE) {
          // every lane: the stage's scales into this CTA's own slots (zero past M)
          float* scs = reinterpret_cast<float*>(ring + stage * C::STAGE + C::SCL_OFF);
          const int mt0 = (u / p.n_tiles) * PN;  // the pair tile's first token
#pragma unroll
          for (int j = 0; j < KS; ++j) {
            const float* sxk = p.sx + static_cast<int64_t>(ks * KS + j) * p.ldsx;
            const float* swk = p.sw + static_cast<int64_t>(ks * KS + j) * p.ldsw;
            float* ssl = scs + j * 256;
            for (int i = lane; i < PN; i += 32) {
              const int m = mt0 + i;
              cp_async_4(&ssl[i], sxk + ((m < p.M ? m : p.M - 1) >> p.gM_shift), m < p.M ? 4u : 0u);
            }
            if (p.gN_shift == 0) {
              for (int i = lane; i < BM; i += 32) cp_async_4(&ssl[PN + i], swk + n_tile * BM + i, 4u);
            } else if (lane == 0) {
              cp_async_4(&ssl[PN], swk + ((n_tile * BM) >> p.gN_shift), 4u);
            }
          }
          cp_async_arrive(&sfull[stage]);
        }
      }
    }
    if (lane == 0) {
      if (!ok) atomicOr(p.err, DEVERR_TIMEOUT_PRODUCER);
      // Before leaving: the MMA has released every stage this warp filled (so its
      // copies have landed and nothing writes this CTA's shared memory later).
      // Only the last use of a slot may be waited on.
      const int64_t fmax = flat - 1;
      for (int64_t f = fmax; f >= 0 && f > fmax - C::STAGES; --f) {
        if (f % PRODUCERS != warp) continue;
        (void)mbar_wait<true>(&empty[f % C::STAGES], static_cast<uint32_t>((f / C::STAGES) & 1));
      }
    }
  } else if (warp == MMA_WARP) {
    // ----------------------------------------------------------- MMA issuer
    if (leader && lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3(2 * BM, PN, true);
      constexpr uint32_t idesc_side = idesc_bf16(2 * BM, PN);
      constexpr uint64_t STAGE_DESC = C::STAGE >> 4;
      const uint32_t ring_u32 = smem_u32(ring);
      const uint64_t a_desc0 = smem_desc(ring_u32 + C::A_OFF, 16, 512, SWZ_64B);
      const uint64_t m_desc0 = smem_desc(ring_u32 + C::META_OFF, 128, 128, SWZ_NONE);
      const uint64_t b_desc0 = smem_desc(ring_u32 + C::B_OFF, 16, 1024, SWZ_128B);
      const uint64_t w2_desc0 = smem_desc(ring_u32, 16, 1024, SWZ_128B);
      const uint64_t x2_desc0 = smem_desc(ring_u32 + SIDE_W2_BYTES, 16, 1024, SWZ_128B);
      uint32_t stage = 0, phase = 0, meta_ctr = 0, acc_cnt = 0;
      bool ok = true;
      for (int u = pair; u < num_units && ok; u += npairs) {
        if (!PROMOTE) {
          if (!mbar_wait<true>(acce, (acc_cnt & 1) ^ 1)) { ok = false; break; }
          tc_fence_after();
        }
        for (int ks = SIDE ? -1 : 0; ks < k_stages; ++ks) {
          if (!mbar_wait<true>(&full[stage], phase)) { ok = false; break; }
          tc_fence_after();
          const uint64_t off = stage * STAGE_DESC;
          if (SIDE && ks < 0) {
            // X2 W2^T into the side accumulator: r / 16 bf16 MMAs, +32 B per 16 of K
            for (int j = 0; j < p.side_ksteps; ++j)
              mma_bf16_pair(tbase + SIDE_COL, w2_desc0 + off + 2 * j, x2_desc0 + off + 2 * j, idesc_side,
                            j > 0 ? 1u : 0u);
          } else {
            const int nsub = min(KS, p.k_tiles - ks * KS);
#pragma unroll
            for (int j = 0; j < KS; ++j) {
              if (j < nsub) {
                // promotion: each K block's partial into its own accumulator,
                // once both epilogues have read that accumulator's last partial
                uint32_t d = tbase, b = 0;
                if (PROMOTE) {
                  b = acc_cnt % NACC;
                  if (!mbar_wait<true>(&acce[b], ((acc_cnt / NACC) & 1) ^ 1)) { ok = false; break; }
                  tc_fence_after();
                  d = tbase + b * PN;
                }
                const uint32_t mcol = tbase + C::META_BASE + 4 * (meta_ctr & (C::META_RING - 1));
                ++meta_ctr;
                tmem_cp_128x128b_pair(mcol, m_desc0 + off + j * (META_STAGE >> 4));
                const uint64_t aj = a_desc0 + off + j * (A_STAGE >> 4);
                const uint64_t bj = b_desc0 + off + j * (C::P_B >> 4);
                mma_sp_e4m3_pair(d, aj, bj, mcol, idesc, (!PROMOTE && (ks != 0 || j != 0)) ? 1u : 0u);
                mma_sp_e4m3_pair(d, aj + 2, bj + 4, mcol + 2, idesc, 1u);  // +32 B of A, +64 B of B
                if (PROMOTE) {
                  mma_commit_pair(&accf[b], 3);
                  ++acc_cnt;
                }
              }
            }
          }
          if (!ok) break;
          mma_commit_pair(&empty[stage], 3);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if (!PROMOTE) {
          mma_commit_pair(accf, 3);
          ++acc_cnt;
        }
      }
      if (!ok) atomicOr(p.err, DEVERR_TIMEOUT_MMA);
      mma_commit_pair(drain, 1);  // every MMA issued must finish before TMEM is freed
      (void)mbar_wait<true>(drain, 0);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int ew = warp - EPI_WARP0;              // 0..7
    const int q = warp & 3;                       // TMEM lane quadrant this warp may access
    const int half = ew >> 2;                     // token chunks half, half + 2, half + 4, ...
    const int row = 32 * q + lane;                // weight row within this CTA's 128
    const int et = threadIdx.x - 32 * EPI_WARP0;  // 0..EPI_THREADS-1
    const uint32_t lane_base = tbase + (static_cast<uint32_t>(32 * q) << 16);
    const uint32_t acce_leader = cluster_addr(acce, 0);
    uint32_t acc_cnt = 0, e_stage = 0, e_phase = 0;
    bool ok = true;
    for (int u = pair; u < num_units && ok; u += npairs) {
      const bool last = u + npairs >= num_units;  // this CTA's final tile: the ring is free afterwards
      const int n0 = (2 * (u % p.n_tiles) + static_cast<int>(rank)) * BM;  // this CTA's channels
      const int m0 = (u / p.n_tiles) * PN;                                  // the tile's tokens
      const int n = n0 + row;
      if (et == 0) bulk_wait_read_all();  // the previous tile's stores have read the staging buffer
      if constexpr (PROMOTE) {
        // each K block's partial, times its sx sw, is added into fp32
        // registers: chunk i of this warp covers tokens CHUNK (half + 2 i) + [0, CHUNK)
        float acc[C::COLS];
#pragma unroll
        for (int i = 0; i < C::COLS; ++i) acc[i] = 0.0f;
        const bool per_row_w = p.gN_shift == 0;  // gN = 1: weight scale varies by row
        for (int ks = 0; ks < k_stages; ++ks) {
          // polls (a sleeping wait wakes later, and this warp is the pipeline's slowest stage)
          if (ok && !mbar_wait<false>(&sfull[e_stage], e_phase)) ok = false;  // the stage's scales landed
#pragma unroll
          for (int j = 0; j < KS; ++j) {
            const uint32_t b = acc_cnt % NACC;
            const float* ssl = reinterpret_cast<const float*>(ring + e_stage * C::STAGE + C::SCL_OFF) + j * 256;
            if (ok && !mbar_wait<false>(&accf[b], (acc_cnt / NACC) & 1)) ok = false;
            ok = __all_sync(0xFFFFFFFFu, ok);
            uint32_t v[C::COLS];
            if (ok) {
              tc_fence_after();
#pragma unroll
              for (int i = 0; i < C::NCHUNK; ++i)
                tmem_load_n<CHUNK>(lane_base + b * PN + CHUNK * (half + 2 * i), v + CHUNK * i);
              tmem_ld_wait();
              tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(acce_leader + 8u * b);  // the partial is in registers
            if (ok) {
              const float rowf = per_row_w ? ssl[PN + row] : ssl[PN];
#pragma unroll
              for (int i = 0; i < C::NCHUNK; ++i)
#pragma unroll
                for (int jj = 0; jj < CHUNK; jj += 4) {
                  const float4 s4 = *reinterpret_cast<const float4*>(ssl + CHUNK * (half + 2 * i) + jj);
                  const int c = CHUNK * i + jj;
                  const float2 s01 = __fmul2_rn(make_float2(s4.x, s4.y), make_float2(rowf, rowf));
                  const float2 s23 = __fmul2_rn(make_float2(s4.z, s4.w), make_float2(rowf, rowf));
                  ffma2(acc[c], acc[c + 1], __uint_as_float(v[c]), __uint_as_float(v[c + 1]), s01.x, s01.y);
                  ffma2(acc[c + 2], acc[c + 3], __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]), s23.x, s23.y);
                }
            }
            ++acc_cnt;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[e_stage]);  // this warp is done with the stage's scales
          if (++e_stage == C::STAGES) { e_stage = 0; e_phase ^= 1; }
        }
        if (epilogue_bar_any(!ok)) { ok = false; break; }
        // the whole tile through the staging buffer: [channel half][PN tokens][64 channels] bf16
        uint16_t* out_row = reinterpret_cast<uint16_t*>(out_tile) + (row >> 6) * (PN * 64) + (row & 63);
        const float bn = bias_of(p, n0 + row);
#pragma unroll
        for (int i = 0; i < C::NCHUNK; ++i)
#pragma unroll
          for (int jj = 0; jj < CHUNK; jj += 4) {
            const int c = CHUNK * i + jj;
            st_bf16x4(out_row + (CHUNK * (half + 2 * i) + jj) * 64, 64, bf16x2_rn(acc[c] + bn, acc[c + 1] + bn),
                      bf16x2_rn(acc[c + 2] + bn, acc[c + 3] + bn));
          }
        fence_proxy_async_smem();
        epilogue_bar();
        if (et == 0) {
          tma_store_2d(&tm_y, out_tile, n0, m0);
          tma_store_2d(&tm_y, out_tile + PN * 128, n0 + 64, m0);
          bulk_commit();
        }
        continue;
      }
      if (et < PN) {
        const int m = m0 + et;
        scl[et] = m < p.M ? __ldg(&p.sx[m >> p.gM_shift]) : 0.0f;
      }
      // loaded before the accumulator is waited on, so that nothing is
      // outstanding when the accumulator is released (a release arrive waits)
      const float swr = __ldg(&p.sw[n >> p.gN_shift]);
      const float bn = bias_of(p, n);
      if (!mbar_wait<true>(accf, acc_cnt & 1)) ok = false;
      if (epilogue_bar_any(!ok)) { ok = false; break; }
      tc_fence_after();
      if constexpr (SIDE) {
      // bf16 results of this thread's row, two tokens per word: chunk i covers
      // tokens CHUNK * (half + 2 i) + [0, CHUNK)
      uint32_t pk[C::COLS / 2];
#pragma unroll
      for (int i = 0; i < C::NCHUNK; ++i) {
        const uint32_t col = lane_base + CHUNK * (half + 2 * i);
        uint32_t v[CHUNK], s2[CHUNK];
        tmem_load_n<CHUNK>(col, v);
        tmem_load_n<CHUNK>(col + SIDE_COL, s2);
        tmem_ld_wait();
        const float* sc = scl + CHUNK * (half + 2 * i);
#pragma unroll
        for (int j = 0; j < CHUNK; j += 4) {
          const uint2 w = scale4_pack<true>(sc + j, swr, v + j, s2 + j, bn);
          pk[(CHUNK * i + j) / 2] = w.x;
          pk[(CHUNK * i + j) / 2 + 1] = w.y;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(acce_leader);  // the next tile's MMAs may overwrite TMEM
      ++acc_cnt;
      if (last) {
        // whole tile through the idle ring: [channel half][PN tokens][64 channels] bf16
        uint16_t* ring_row = reinterpret_cast<uint16_t*>(ring) + (row >> 6) * (PN * 64) + (row & 63);
#pragma unroll
        for (int i = 0; i < C::NCHUNK; ++i)
#pragma unroll
          for (int j = 0; j < CHUNK; j += 4)
            st_bf16x4(ring_row + (CHUNK * (half + 2 * i) + j) * 64, 64, pk[(CHUNK * i + j) / 2],
                      pk[(CHUNK * i + j) / 2 + 1]);
        fence_proxy_async_smem();
        epilogue_bar();
        if (et == 0) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int t = 0; t < PN; t += C::OUT_TOKENS)
              tma_store_2d(&tm_y, ring + c * (PN * 128) + t * 128, n0 + 64 * c, m0 + t);
          bulk_commit();
        }
      } else {
        // passes of OUT_TOKENS tokens through the staging buffer; in pass s
        // every warp stores its chunk s (tokens OUT_TOKENS s + CHUNK half + [0, CHUNK))
        uint16_t* out_row = reinterpret_cast<uint16_t*>(out_tile) + (row >> 6) * (C::OUT_TOKENS * 64) + (row & 63);
#pragma unroll
        for (int s = 0; s < C::NPASS; ++s) {
#pragma unroll
          for (int j = 0; j < CHUNK; j += 4)
            st_bf16x4(out_row + (CHUNK * half + j) * 64, 64, pk[(CHUNK * s + j) / 2], pk[(CHUNK * s + j) / 2 + 1]);
          fence_proxy_async_smem();
          epilogue_bar();
          if (et == 0) {
            tma_store_2d(&tm_y, out_tile, n0, m0 + C::OUT_TOKENS * s);
            tma_store_2d(&tm_y, out_tile + C::OUT_TOKENS * 128, n0 + 64, m0 + C::OUT_TOKENS * s);
            bulk_commit();
            if (s < C::NPASS - 1) bulk_wait_read_all();
          }
          if (s < C::NPASS - 1) epilogue_bar();
        }
      }
      } else {
      uint32_t v[C::COLS];  // chunk i of this warp: tokens CHUNK * (half + 2 i) + [0, CHUNK)
#pragma unroll
      for (int i = 0; i < C::COLS / CHUNK; ++i) tmem_load_n<CHUNK>(lane_base + CHUNK * (half + 2 * i), v + CHUNK * i);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(acce_leader);  // the next tile's MMAs may overwrite TMEM
      ++acc_cnt;
      if (last) {
        // whole tile through the idle ring: [channel half][PN tokens][64 channels] bf16
        uint16_t* ring_row = reinterpret_cast<uint16_t*>(ring) + (row >> 6) * (PN * 64) + (row & 63);
#pragma unroll
        for (int i = 0; i < C::COLS / CHUNK; ++i) {
          const int t0 = CHUNK * (half + 2 * i);
#pragma unroll
          for (int j = 0; j < CHUNK; j += 4)
            scale4_store<false>(scl + t0 + j, swr, v + CHUNK * i + j, nullptr, bn, ring_row + (t0 + j) * 64, 64);
        }
        fence_proxy_async_smem();
        epilogue_bar();
        if (et == 0) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int t = 0; t < PN; t += C::OUT_TOKENS)
              tma_store_2d(&tm_y, ring + c * (PN * 128) + t * 128, n0 + 64 * c, m0 + t);
          bulk_commit();
        }
      } else {
        // NPASS passes of OUT_TOKENS = 2 CHUNK tokens through the staging buffer;
        // in pass s every warp converts its chunk s (tokens OUT_TOKENS s + CHUNK half + [0, CHUNK))
        uint16_t* out_row = reinterpret_cast<uint16_t*>(out_tile) + (row >> 6) * (C::OUT_TOKENS * 64) + (row & 63);
#pragma unroll
        for (int s = 0; s < C::NPASS; ++s) {
          const int t0 = C::OUT_TOKENS * s + CHUNK * half;
#pragma unroll
          for (int j = 0; j < CHUNK; j += 4)
            scale4_store<false>(scl + t0 + j, swr, v + CHUNK * s + j, nullptr, bn, out_row + (CHUNK * half + j) * 64,
                                64);
          fence_proxy_async_smem();
          epilogue_bar();
          if (et == 0) {
            tma_store_2d(&tm_y, out_tile, n0, m0 + C::OUT_TOKENS * s);
            tma_store_2d(&tm_y, out_tile + C::OUT_TOKENS * 128, n0 + 64, m0 + C::OUT_TOKENS * s);
            bulk_commit();
            if (s < C::NPASS - 1) bulk_wait_read_all();
          }
          if (s < C::NPASS - 1) epilogue_bar();
        }
      }
      }
    }
    if (et == 0) bulk_wait_all();
    if (!ok) atomicOr(p.err, DEVERR_TIMEOUT_EPILOGUE);
  }

  pdl_trigger();  // only teardown is left: the next kernel may begin launching
  tc_fence_before();
  cluster_sync();  // no CTA leaves while its peer may still signal it or read its shared memory
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, 512);
  }
}

}  // namespace

bool pair_gemm_applies(int64_t M, int64_t N, int64_t K, bool plain, int64_t r) {
  // 256-token tiles (240 with the side GEMM) pay off from a little under one
  // full tile; TMA row coordinates of the tiled weight views must fit in int32
  return plain && r <= 64 && M > 192 && N % (2 * BM) == 0 && (N / 256) * (K + BK) < (int64_t(1) << 31);
}

bool pair_promote_applies(int64_t M, int64_t N, int64_t K, int64_t r) {
  // 128-token pair tiles with a partial per K block; stages hold whole pairs of K blocks
  return r == 0 && M > 64 && N % (2 * BM) == 0 && (K / BK) % KS == 0 && (N / 256) * (K + BK) < (int64_t(1) << 31);
}

namespace {

template <int PN, bool SIDE, bool PROMOTE>
sp24_status launch_pair(const DeviceInfo* dev, const void* Xq, int64_t ldx, const void* Y, int64_t ldy,
                        const void* X2, const void* W2, int64_t r, const GemmArgs& args_in, cudaStream_t stream) {
  using C = PairCfg<PN, SIDE, PROMOTE>;
  GemmArgs a = args_in;
  const int64_t M = a.M, N = a.N, K = a.K;
  a.m_tiles = static_cast<int>((M + PN - 1) / PN);
  a.n_tiles = static_cast<int>(N / (2 * BM));
  a.k_tiles = static_cast<int>(K / BK);
  a.side_ksteps = SIDE ? static_cast<int>(r / 16) : 0;
  CUtensorMap tm_x, tm_v, tm_m, tm_y, tm_w2, tm_x2;
  sp24_status st = make_tmap_2d(&tm_x, Xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, ldx, BK, C::HALF_N,
                                CU_TENSOR_MAP_SWIZZLE_128B);
  // tiled weight storage as 128-byte rows: a values tile is 64 rows, a metadata tile 16
  if (st == SP24_OK)
    st = make_tmap_2d(&tm_v, a.values, CU_TENSOR_MAP_DATA_TYPE_UINT8, 128, N * K / 256, 128, 128, KS * VROWS,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st == SP24_OK)
    st = make_tmap_2d(&tm_m, a.meta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 128, N * K / 1024, 128, 128, KS * MROWS,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st == SP24_OK)
    st = make_tmap_2d(&tm_y, Y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, ldy * 2, 64, C::OUT_TOKENS,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  if (SIDE) {
    // [rows][r] bf16, boxes of 64 columns (zero fill past r), 128-byte swizzle
    if (st == SP24_OK)
      st = make_tmap_2d(&tm_w2, W2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, r, N, r * 2, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == SP24_OK)
      st = make_tmap_2d(&tm_x2, X2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, r, M, r * 2, 64, C::HALF_N,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    tm_w2 = tm_x;
    tm_x2 = tm_x;
  }
  if (st != SP24_OK) return st;

  auto kern = sp24_gemm_pair_kernel<PN, SIDE, PROMOTE>;
  static std::atomic<int> max_pairs[64];  // per device: co-resident pairs (0 = not yet known; races are idempotent)
  const int d = dev->ordinal;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int known = max_pairs[d].load(std::memory_order_acquire);
  if (known == 0) {
    if (static_cast<size_t>(C::SMEM) > dev->smem_optin) return SP24_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return SP24_ERR_CUDA;
    cfg.gridDim = dim3(2 * (dev->sm_count / 2), 1, 1);
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess || active < 1) return SP24_ERR_CUDA;
    max_pairs[d].store(active, std::memory_order_release);
    known = active;
  }
  const int units = a.m_tiles * a.n_tiles;
  const int pairs = units < known ? units : known;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, kern, tm_x, tm_v, tm_m, tm_y, tm_w2, tm_x2, a) != cudaSuccess) return SP24_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SP24_OK : SP24_ERR_CUDA;
}

}  // namespace

// Token tile of the plain kernel: 256, or 240 where that takes fewer
// tile-widths of time, counting every round of tiles over the SM pairs as
// a full one (M = 2048: 144 tiles of 240 in two rounds against 128 of 256).
int pair_token_tile(int64_t M, int64_t N, int sm_count) {
  const int64_t pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
  auto cost = [&](int64_t pn) { return ((M + pn - 1) / pn * (N / 256) + pairs - 1) / pairs * pn; };
  return cost(240) < cost(256) ? 240 : 256;
}

sp24_status launch_pair_gemm(const DeviceInfo* dev, const void* Xq, int64_t ldx, const void* Y, int64_t ldy,
                             const void* X2, const void* W2, int64_t r, const GemmArgs& args, cudaStream_t stream) {
  if (r > 0) return launch_pair<240, true, false>(dev, Xq, ldx, Y, ldy, X2, W2, r, args, stream);
  if (pair_token_tile(args.M, args.N, dev->sm_count) == 240)
    return launch_pair<240, false, false>(dev, Xq, ldx, Y, ldy, X2, W2, 0, args, stream);
  return launch_pair<256, false, false>(dev, Xq, ldx, Y, ldy, X2, W2, 0, args, stream);
}

// Token tile of a group-wise pair launch: 112 (four accumulators) where it
// takes no more rounds of tiles over the SM pairs than 128 (three), counting
// a 112-token round at the 0.93 of a 128-token one measured on the 152-SM part
// (N 4096, M 2048: 52.6 against 56.9 us in four rounds each).
int pair_promote_token_tile(int64_t M, int64_t N, int sm_count) {
  const int64_t pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
  auto rounds = [&](int64_t pn) { return ((M + pn - 1) / pn * (N / 256) + pairs - 1) / pairs; };
  return rounds(112) * 93 < rounds(128) * 100 ? 112 : 128;
}

sp24_status launch_pair_promote(const DeviceInfo* dev, const void* Xq, int64_t ldx, const void* Y, int64_t ldy,
                                const GemmArgs& args, cudaStream_t stream) {
  if (pair_promote_token_tile(args.M, args.N, dev->sm_count) == 112)
    return launch_pair<112, false, true>(dev, Xq, ldx, Y, ldy, nullptr, nullptr, 0, args, stream);
  return launch_pair<128, false, true>(dev, Xq, ldx, Y, ldy, nullptr, nullptr, 0, args, stream);
}

}  // namespace sp24
