// sp24_gemm.cu -- 2:4 sparse e4m3 GEMM with group-wise scaling and an
// optional fused bf16 side GEMM, for sm_103a.
//
// Math (user view):  Y[m][n] = bf16( sum_kb sx[kb][m/gM] sw[kb][n/gN] P_kb[m][n]
//                                    + sum_j X2[m][j] W2[n][j] ).
// The kernel computes the transposed product Y^T = W . X^T so that the
// sparse weight is the row-major sparse A operand of the tensor core and the
// token-major activations are the K-major B operand (CUTLASS issue #2029,
// klevzoff's swap+transpose answer); a weight row is a TMEM lane and a token
// is a TMEM column.  Row-major Y is column-major Y^T, so nothing is moved.
//
// Structure (one CTA per SM, 11 warps):
//   warps 0-1   producers, taking pipeline stages in turn: per stage, KS
//               128-wide K steps of kept values (128 rows x 64 B each,
//               64-byte swizzle) and metadata (128 rows x 16 B) in two bulk
//               copies, and KS activation boxes (BN rows x 128 B, 128-byte
//               swizzle) by TMA, into one stage of a shared-memory ring.
//   warp 2      TMEM allocation and the single-thread MMA issuer: copies each
//               K step's metadata into TMEM (tcgen05.cp, lane = weight row)
//               and issues two sparse tcgen05.mma (K = 64 each) per K step.
//   warps 3-10  epilogue: tcgen05.ld of the fp32 accumulator, scale, add the
//               side accumulator and the bias, round to bf16, TMA store
//               (rows past M clipped by the tensor map).
// Schedules (the host picks one per call): whole tiles dealt round-robin to
// persistent CTAs; stream-K over all tiles' stages with partials exchanged
// through a workspace; or a cluster split, each tile's K range cut across a
// 2- or 4-CTA cluster whose peers send their partials into the leader CTA's
// shared memory.  Large token counts use the SM-pair kernel instead
// (sp24_gemm_pair.cu).
// Scale promotion (gK = 128, CUTLASS PR #2095's per-K-tile promotion): every
// 128-wide K step is its own scale block, so each stage's partial product
// lands in its own TMEM buffer (ring of NACC) and the epilogue folds it into
// register accumulators with sx * sw while the tensor core fills the next.
// Partial token tiles: TMA zero-fills rows past M and the epilogue skips them
// (PR #2095, predication of partial tiles).
// Side GEMM (CUTLASS issue #2058, Y = X1 W1^T + X2 W2^T in one kernel): after
// the sparse K loop the MMA thread issues bf16 tcgen05.mma over r <= 64 into
// a second accumulator that the epilogue adds after scaling.
#include <cuda_bf16.h>
#include <atomic>
#include <chrono>
#include <mutex>
#include "sp24_gemm_common.cuh"
#include "sp24_internal.cuh"
#include "sp24_ptx.cuh"

namespace sp24 {
namespace {

// A pipeline stage carries KS consecutive 128-K sub-tiles: the kept values
// of all KS (one contiguous copy), their metadata (one copy), then KS
// activation boxes.  Small token tiles use KS > 1 so that each barrier
// round trip and metadata copy is amortised over more MMAs.
template <int BN, bool PROMOTE, bool SIDE, bool SPLIT, int KS, bool CSPLIT = false>
struct Cfg {
  static constexpr int B_SUB = BN * BK;               // e4m3 activations of one sub-tile, 128 B per token row
  static constexpr int A_OFF = 0;
  static constexpr int META_OFF = KS * A_STAGE;
  static constexpr int B_OFF = KS * (A_STAGE + META_STAGE);
  static constexpr int SCL_OFF = B_OFF + KS * B_SUB;
  static constexpr int SCL_STAGE = PROMOTE ? KS * 1024 : 0;  // per K block of the stage: sx[BN] then sw[128]
  static constexpr int STAGE = SCL_OFF + SCL_STAGE;
  static constexpr int LOAD_BYTES = KS * (A_STAGE + META_STAGE + B_SUB);
  static constexpr int SIDE_BYTES = SIDE ? (BM * 128 + BN * 128) : 0;
  // bf16 output staged for the TMA store: the whole tile, or (BN = 256) half of it at a time
  static constexpr int OUT_TOKENS = BN > 128 ? BN / 2 : BN;
  static constexpr int OUT_BYTES = OUT_TOKENS * BM * 2;
  static constexpr int NACC = BN > 128 ? 1 : ((PROMOTE && !SIDE && 3 * BN <= META_COL0) ? 3 : 2);
  static constexpr int SCALE_BYTES = 4 * BN;
  // cluster split: the leader CTA receives its peers' fp32 partials [peer][col][row]
  static constexpr int CS_PEERS = CSPLIT ? (BN <= 32 ? 3 : 1) : 0;
  static constexpr int PART_BYTES = CS_PEERS * BN * BM * 4;
  static constexpr int FIXED = 1024 + SIDE_BYTES + OUT_BYTES + SCALE_BYTES + PART_BYTES + BAR_BYTES;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - FIXED) / STAGE;
  static constexpr int STAGES_CAP = META_SLOTS / KS;  // metadata ring covers every sub-tile in flight
  static constexpr int STAGES = STAGES_FIT < STAGES_CAP ? STAGES_FIT : STAGES_CAP;
  static constexpr int SMEM = FIXED + STAGES * STAGE;
  static constexpr int COLS = BN / 2;  // accumulator columns (tokens) per epilogue warp
  static_assert(STAGE % 1024 == 0 && B_OFF % 1024 == 0 && B_SUB % 1024 == 0, "1024-byte swizzle alignment");
  static_assert(STAGES >= 2, "need at least two stages");
  static_assert(NACC * BN + (SIDE ? BN : 0) <= META_COL0, "TMEM columns");
  static_assert(COLS % 8 == 0, "epilogue chunking");
  static_assert(BN <= 128 || (!PROMOTE && !SIDE), "256-token tiles: plain per-tensor-K scaling only");
  static_assert(!PROMOTE || (BN <= 128 && KS <= 2), "a scale slot holds BN + 128 floats per K block");
  static_assert(!SPLIT || (!PROMOTE && !SIDE && BN <= 128), "stream-K: plain per-tensor-K scaling only");
  static_assert(!CSPLIT || (!PROMOTE && !SIDE && !SPLIT && BN <= 64), "cluster split: plain small-token tiles only");
};

// Work schedule.  A tile is (problem of the batch, token tile, weight tile),
// numbered weight tile fastest.  Without stream-K the persistent CTAs take
// whole tiles round-robin.  With stream-K (SPLIT) the S stages of all tiles'
// stage sequences are dealt out to the C CTAs in contiguous ranges, the
// first S mod C CTAs taking one stage more than the rest, and each range is
// cut where the tile changes: a piece that starts at a tile's first stage
// completes that tile (adding the partials of the CTAs that hold its later
// stages, which start their ranges with them); any other piece is published
// as this CTA's partial.  The host keeps S (and the tile count) below 2^31,
// so all of this is 32-bit arithmetic.  With a cluster split (MODE 2) each
// cluster of C CTAs takes one tile and CTA rank r its stages
// [r kst / C, (r + 1) kst / C); rank 0 completes the tile with the other
// ranks' partials, which arrive in its shared memory.
struct Unit {
  int b, m_tile, n_tile, kt0, kt1;
  uint32_t tile;
  int role;  // 0: a whole tile; 1: a tile's first stages, completes it; 2: later stages, published;
             // cluster split: 3 the leader's stages, completes the tile; 4 a peer's stages, sent to the leader
};
struct WorkIter {
  uint32_t pos, end;
};
template <int MODE>  // 0: whole tiles, 1: stream-K, 2: cluster split
__device__ __forceinline__ WorkIter work_begin(const GemmArgs& p) {
  if (MODE == 2) {
    const uint32_t c = cluster_id_x();
    return {c, c + 1};
  }
  if (MODE == 1) {
    const uint32_t units = static_cast<uint32_t>(p.sk_units), q = units / gridDim.x, r = units % gridDim.x;
    const uint32_t c = blockIdx.x;
    const uint32_t begin = c * q + (c < r ? c : r);
    return {begin, begin + q + (c < r ? 1u : 0u)};
  }
  return {blockIdx.x, static_cast<uint32_t>(p.L) * static_cast<uint32_t>(p.m_tiles) * static_cast<uint32_t>(p.n_tiles)};
}
template <int MODE, int KS>
__device__ __forceinline__ bool work_next(const GemmArgs& p, WorkIter& w, Unit& t) {
  if (w.pos >= w.end) return false;
  if (MODE == 2) {
    const uint32_t kst = static_cast<uint32_t>(p.kst), r = cluster_rank(), cs = cluster_nrank();
    t.tile = w.pos;
    w.pos = w.end;
    t.kt0 = static_cast<int>(r * kst / cs) * KS;
    t.kt1 = min(static_cast<int>((r + 1) * kst / cs) * KS, p.k_tiles);
    t.role = r == 0 ? 3 : 4;
  } else if (MODE == 1) {
    const uint32_t kst = static_cast<uint32_t>(p.kst);
    t.tile = w.pos / kst;
    const uint32_t s0 = w.pos - t.tile * kst;
    const uint32_t s1 = min(kst, s0 + (w.end - w.pos));
    w.pos += s1 - s0;
    t.kt0 = static_cast<int>(s0) * KS;
    t.kt1 = min(static_cast<int>(s1) * KS, p.k_tiles);
    t.role = (s0 == 0 && s1 == kst) ? 0 : (s0 == 0 ? 1 : 2);
  } else {
    t.tile = w.pos;
    w.pos += gridDim.x;
    t.kt0 = 0;
    t.kt1 = p.k_tiles;
    t.role = 0;
  }
  const uint32_t nt = static_cast<uint32_t>(p.n_tiles), mt = static_cast<uint32_t>(p.m_tiles);
  const uint32_t rest = t.tile / nt;
  t.n_tile = static_cast<int>(t.tile - rest * nt);
  const uint32_t b = rest / mt;
  t.m_tile = static_cast<int>(rest - b * mt);
  t.b = static_cast<int>(b);
  return true;
}
// The CTA whose stream-K range holds stage s (the inverse of work_begin).
__device__ __forceinline__ int sk_owner(const GemmArgs& p, uint32_t s) {
  const uint32_t units = static_cast<uint32_t>(p.sk_units), q = units / gridDim.x, r = units % gridDim.x;
  const uint32_t big = r * (q + 1);  // stages held by the CTAs with one stage more
  return static_cast<int>(s < big ? s / (q + 1) : r + (s - big) / q);
}

template <int BN, bool PROMOTE, bool SIDE, bool SPLIT, int KS, bool CSPLIT = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    sp24_gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w2,
                     const __grid_constant__ CUtensorMap tm_x2, const __grid_constant__ CUtensorMap tm_y,
                     const GemmArgs p) {
  using C = Cfg<BN, PROMOTE, SIDE, SPLIT, KS, CSPLIT>;
  constexpr int SCHED = SPLIT ? 1 : (CSPLIT ? 2 : 0);
  constexpr int STAGES = C::STAGES;
  constexpr int NACC = C::NACC;
  constexpr int COLS = C::COLS;
  constexpr int CH = COLS >= 16 ? 16 : COLS;  // columns per TMEM load
  constexpr int SK_GRP = COLS <= 8 ? 8 : 64 / COLS;  // stream-K partials gathered ahead (64 floats)
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base by pointer arithmetic on the shared array, so that
  // accesses through it compile to shared-memory instructions
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = sm;
  uint8_t* side_w2 = sm + STAGES * C::STAGE;
  uint8_t* side_x2 = side_w2 + BM * 128;
  uint8_t* out_tile = sm + STAGES * C::STAGE + C::SIDE_BYTES;      // [2 halves][tokens][64 channels] bf16
  float* scl = reinterpret_cast<float*>(out_tile + C::OUT_BYTES);  // per-tile token scales [BN]
  float* part = reinterpret_cast<float*>(out_tile + C::OUT_BYTES + C::SCALE_BYTES);  // cluster split, leader
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_tile + C::OUT_BYTES + C::SCALE_BYTES + C::PART_BYTES);
  uint64_t* full = bars;                   // [STAGES] loads -> MMA
  uint64_t* empty = bars + MAX_STAGES;     // [STAGES] MMA (and promotion epilogue) -> loads, cluster-wide
  uint64_t* accf = bars + 2 * MAX_STAGES;  // [NACC]  MMA -> epilogue
  uint64_t* acce = accf + 3;               // [NACC]  epilogue -> MMA
  uint64_t* sidef = acce + 3;              // side operands loaded
  uint64_t* sidee = sidef + 1;             // side operands consumed
  uint64_t* saccf = sidee + 1;             // side accumulator ready
  uint64_t* sacce = saccf + 1;             // side accumulator drained
  uint64_t* drain = sacce + 1;             // MMA drain on abort
  uint64_t* pfull = drain + 1;             // cluster split, leader: every peer partial landed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(pfull + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1 + (PROMOTE ? 32 : 0));
      mbar_init(&empty[i], 1 + (PROMOTE ? EPI_WARPS : 0));
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], EPI_WARPS);  // one arrival per epilogue warp
    }
    mbar_init(sidef, 1);
    mbar_init(sidee, 1);
    mbar_init(saccf, 1);
    mbar_init(sacce, EPI_WARPS);
    mbar_init(drain, 1);
    if (CSPLIT) mbar_init(pfull, 1);
    fence_mbar_init();
    // the leader expects every peer's partial (st.async bytes) on pfull
    if (CSPLIT && cluster_rank() == 0) mbar_arrive_expect_tx(pfull, (cluster_nrank() - 1) * (BN * BM * 4));
  }
  if (warp == MMA_WARP + 1 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_y);
    if (SIDE) {
      tma_prefetch_desc(&tm_w2);
      tma_prefetch_desc(&tm_x2);
    }
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  if constexpr (CSPLIT)
    cluster_sync();  // the leader's pfull exists before any peer stores to it
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  if (BN <= 16 && warp == 0 && lane == 0) {
    // Decode tiles: while the previous kernel finishes, the weight bytes of the
    // first 8 K blocks of this CTA's first unit into L2 (measured: 0.6 us of a
    // 15 us weight stream; no gain with wider token tiles, or with more bytes)
    WorkIter w0 = work_begin<SCHED>(p);
    Unit t0;
    if (work_next<SCHED, KS>(p, w0, t0)) {
      const int kend = min(t0.kt1, t0.kt0 + 8);
      const uint8_t* vsrc = p.values + t0.b * p.bs_values + static_cast<int64_t>(t0.n_tile) * p.k_tiles * A_STAGE;
      const uint8_t* msrc = p.meta + t0.b * p.bs_meta + static_cast<int64_t>(t0.n_tile) * p.k_tiles * META_STAGE;
      for (int kt = t0.kt0; kt < kend; kt += 4) {
        const int nk = min(4, kend - kt);
        bulk_prefetch_l2(vsrc + static_cast<int64_t>(kt) * A_STAGE, nk * A_STAGE);
        bulk_prefetch_l2(msrc + static_cast<int64_t>(kt) * META_STAGE, nk * META_STAGE);
      }
    }
  }
  pdl_wait();  // the previous kernel's writes are visible from here on

  if (warp < PRODUCERS) {
    // ----------------------------------------------------------- producers
    // Every mbarrier operation costs its thread a round trip, so stages are
    // dealt out to PRODUCERS warps in turn (warp p takes flat stage indices
    // p, p + PRODUCERS, ...).  Lane 0 issues the bulk/TMA copies; with
    // promotion all 32 lanes also copy the stage's scale vectors (cp.async,
    // zero-filled past M).
    const int pw = warp;
    int64_t flat = 0;  // stage index over this CTA's whole tile sequence
    uint32_t side_phase = 0;
    bool ok = true;
    WorkIter work = work_begin<SCHED>(p);
    Unit t;
    while (ok && work_next<SCHED, KS>(p, work, t)) {
      const int n_tile = t.n_tile;
      const int n0 = n_tile * BM;
      const int m0 = t.m_tile * BN;
      const uint8_t* vsrc = p.values + t.b * p.bs_values + static_cast<int64_t>(n_tile) * p.k_tiles * A_STAGE;
      const uint8_t* msrc = p.meta + t.b * p.bs_meta + static_cast<int64_t>(n_tile) * p.k_tiles * META_STAGE;
      for (int kt = t.kt0; kt < t.kt1; kt += KS, ++flat) {
        if (flat % PRODUCERS != pw) continue;
        const uint32_t stage = static_cast<uint32_t>(flat % STAGES);
        const uint32_t phase = static_cast<uint32_t>((flat / STAGES) & 1);
        const bool got = mbar_wait(&empty[stage], phase ^ 1);
        if (!__all_sync(0xFFFFFFFFu, got)) { ok = false; break; }
        uint8_t* sA = ring + stage * C::STAGE;
        // A fault-test build (SP24_FAULT_WITHHOLD_FIRST_STAGE, which the
        // library itself never defines) issues nothing for the CTA's first
        // stage: no copies are in flight for it, and the MMA thread's bounded
        // wait for it runs out.  The tests use it to check the give-up path.
#ifdef SP24_FAULT_WITHHOLD_FIRST_STAGE
        const bool issue = flat != 0;
#else
        constexpr bool issue = true;
#endif
        if (lane == 0 && issue) {
          mbar_arrive_expect_tx(&full[stage], C::LOAD_BYTES);
          bulk_load(sA + C::A_OFF, vsrc + static_cast<int64_t>(kt) * A_STAGE, KS * A_STAGE, &full[stage]);
          bulk_load(sA + C::META_OFF, msrc + static_cast<int64_t>(kt) * META_STAGE, KS * META_STAGE, &full[stage]);
#pragma unroll
          for (int j = 0; j < KS; ++j)
            tma_load_3d(sA + C::B_OFF + j * C::B_SUB, &tm_x, &full[stage], (kt + j) * BK, m0, t.b);
        }
        if (PROMOTE) {
#pragma unroll
          for (int j = 0; j < KS; ++j) {  // the scales of each K block of the stage, in its own slot
            float* ssl = reinterpret_cast<float*>(sA + C::SCL_OFF + j * 1024);
            const float* sxk = p.sx + t.b * p.bs_sx + static_cast<int64_t>(kt + j) * p.ldsx;
            for (int i = lane; i < BN; i += 32) {
              const int m = m0 + i;
              cp_async_4(&ssl[i], sxk + ((m < p.M ? m : p.M - 1) >> p.gM_shift), m < p.M ? 4u : 0u);
            }
            const float* swk = p.sw + t.b * p.bs_sw + static_cast<int64_t>(kt + j) * p.ldsw;
            if (p.gN_shift == 0) {
              for (int i = lane; i < BM; i += 32) cp_async_4(&ssl[BN + i], swk + n0 + i, 4u);
            } else if (lane == 0) {
              cp_async_4(&ssl[BN], swk + (n0 >> p.gN_shift), 4u);
            }
          }
          cp_async_arrive(&full[stage]);
        }
      }
      if (SIDE && ok && pw == 0) {
        const bool got = mbar_wait(sidee, side_phase ^ 1);
        if (!__all_sync(0xFFFFFFFFu, got)) { ok = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(sidef, BM * 128 + BN * 128);
          tma_load_2d(side_w2, &tm_w2, sidef, 0, n0);
          tma_load_2d(side_x2, &tm_x2, sidef, 0, m0);
        }
        side_phase ^= 1;
      }
    }
    if (lane == 0) {
      if (!ok) atomicOr(p.err, DEVERR_TIMEOUT_PRODUCER);
      // Before leaving: every stage this warp issued has landed (so nothing writes
      // this CTA's shared memory later) and its consumers have released it.
      // Only the last use of a slot may be waited on (an older phase of the same
      // parity would not be seen as complete).
      const int64_t fmax = flat - 1;
      for (int64_t f = fmax; f >= 0 && f > fmax - STAGES; --f) {
        if (f % PRODUCERS != pw) continue;
        (void)mbar_wait(&full[f % STAGES], static_cast<uint32_t>((f / STAGES) & 1));
        (void)mbar_wait(&empty[f % STAGES], static_cast<uint32_t>((f / STAGES) & 1));
      }
    }
  } else if (warp == MMA_WARP) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_sp = idesc_e4m3(BM, BN, true);
      constexpr uint32_t idesc_side = idesc_bf16(BM, BN);
      constexpr uint64_t STAGE_DESC = C::STAGE >> 4;  // descriptor start-address units per stage
      // stage-0 descriptors; a stage is a fixed offset in the start-address field
      const uint32_t ring_u32 = smem_u32(ring);
      const uint64_t a_desc0 = smem_desc(ring_u32 + C::A_OFF, 16, 512, SWZ_64B);
      const uint64_t m_desc0 = smem_desc(ring_u32 + C::META_OFF, 128, 128, SWZ_NONE);
      const uint64_t b_desc0 = smem_desc(ring_u32 + C::B_OFF, 16, 1024, SWZ_128B);
      uint32_t stage = 0, phase = 0, side_cnt = 0, meta_ctr = 0;
      uint32_t acc_cnt = 0;
      bool ok = true;
      WorkIter work = work_begin<SCHED>(p);
      Unit t;
      while (ok && work_next<SCHED, KS>(p, work, t)) {
        uint32_t d = 0;
        if (!PROMOTE) {
          const uint32_t b = acc_cnt % NACC;
          if (!mbar_wait(&acce[b], ((acc_cnt / NACC) & 1) ^ 1)) { ok = false; break; }
          tc_fence_after();
          d = tbase + b * BN;
        }
        for (int kt = t.kt0; kt < t.kt1 && ok; kt += KS) {
          if (!mbar_wait(&full[stage], phase)) { ok = false; break; }
          const uint64_t off = stage * STAGE_DESC;
#pragma unroll
          for (int j = 0; j < KS; ++j) {
            uint32_t b = 0;
            if (PROMOTE) {  // each K block's partial goes to its own accumulator buffer
              b = acc_cnt % NACC;
              if (!mbar_wait(&acce[b], ((acc_cnt / NACC) & 1) ^ 1)) { ok = false; break; }
              tc_fence_after();
              d = tbase + b * BN;
            }
            const uint32_t mcol = tbase + META_COL0 + 4 * (meta_ctr & (META_SLOTS - 1));
            ++meta_ctr;
            tmem_cp_128x128b(mcol, m_desc0 + off + j * (META_STAGE >> 4));
            const uint32_t acc0 = PROMOTE ? 0u : ((kt != t.kt0 || j != 0) ? 1u : 0u);
            const uint64_t aj = a_desc0 + off + j * (A_STAGE >> 4);
            const uint64_t bj = b_desc0 + off + j * (C::B_SUB >> 4);
            mma_sp_e4m3(d, aj, bj, mcol, idesc_sp, acc0);
            mma_sp_e4m3(d, aj + 2, bj + 4, mcol + 2, idesc_sp, 1u);  // +32 B of A, +64 B of B
            if (PROMOTE) {
              mma_commit(&accf[b]);
              ++acc_cnt;
            }
          }
          if (!ok) break;
          mma_commit(&empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if (SIDE) {
          if (!mbar_wait(sacce, (side_cnt & 1) ^ 1)) { ok = false; break; }
          if (!mbar_wait(sidef, side_cnt & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t ds = tbase + NACC * BN;
          for (int j = 0; j < p.side_ksteps; ++j) {
            const uint64_t da = smem_desc(smem_u32(side_w2) + 32 * j, 16, 1024, SWZ_128B);
            const uint64_t db = smem_desc(smem_u32(side_x2) + 32 * j, 16, 1024, SWZ_128B);
            mma_bf16(ds, da, db, idesc_side, j > 0);
          }
          mma_commit(sidee);
          mma_commit(saccf);
          ++side_cnt;
        }
        if (!PROMOTE) {
          mma_commit(&accf[acc_cnt % NACC]);
          ++acc_cnt;
        }
      }
      if (!ok) atomicOr(p.err, DEVERR_TIMEOUT_MMA);
      mma_commit(drain);  // every MMA issued so far must finish before TMEM is freed
      (void)mbar_wait(drain, 0);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int ew = warp - EPI_WARP0;          // 0..7
    const int q = warp & 3;                   // TMEM lane quadrant this warp may access
    const int half = ew >> 2;                 // which half of the tile's columns
    const int row = 32 * q + lane;            // weight row (channel) within the tile
    const int et = threadIdx.x - 32 * EPI_WARP0;  // 0..EPI_THREADS-1
    const int c0 = half * COLS;               // first accumulator column (token) of this warp
    const uint32_t lane_base = tbase + (static_cast<uint32_t>(32 * q) << 16);
    // staged output: channel half (row / 64) x tokens x 64 channels
    uint16_t* out_row = reinterpret_cast<uint16_t*>(out_tile) + (row >> 6) * (C::OUT_TOKENS * 64) + (row & 63);
    uint32_t acc_cnt = 0, side_cnt = 0, e_stage = 0, e_phase = 0;
    bool ok = true;
    // stream-K: this launch's epoch (the counter changes only after every CTA
    // of the launch has finished; the previous launch is complete here)
    const unsigned long long epoch = SPLIT ? (*reinterpret_cast<volatile unsigned long long*>(p.sk_word) >> 20) + 1 : 0;
    WorkIter work = work_begin<SCHED>(p);
    Unit t;
    while (ok && work_next<SCHED, KS>(p, work, t)) {
      const int n0 = t.n_tile * BM;
      const int m0 = t.m_tile * BN;
      const int n = n0 + row;
      if (et == 0) bulk_wait_read_all();  // the previous tile's store has read the staging buffer
      if (!PROMOTE) {
        const uint32_t b = acc_cnt % NACC;
        if (et < BN) {
          const int m = m0 + et;
          scl[et] = m < p.M ? __ldg(&p.sx[t.b * p.bs_sx + (m >> p.gM_shift)]) : 0.0f;
        }
        // stream-K, a tile's first stages: gather the other CTAs' partials
        // while this CTA's own stages are still being loaded and multiplied.
        // Those CTAs publish their partials at the start of their ranges, so
        // the waits are usually already over.  One thread per partial watches
        // its flag (the waits overlap); the first SK_GRP partials are read
        // into registers at once, the rest (rare) after the accumulator.
        int nparts = 0;
        float pre[SPLIT ? SK_GRP : 1][SPLIT ? COLS : 1];
        const float* wsp = nullptr;
        if constexpr (SPLIT) {
          if (t.role == 1) {
            const int first = static_cast<int>(blockIdx.x) + 1;
            nparts = sk_owner(p, t.tile * static_cast<uint32_t>(p.kst) + p.kst - 1) + 1 - first;
            bool got = true;
            for (int i = et; i < nparts; i += EPI_THREADS) {
              const uint64_t t0 = globaltimer_ns();
              while (ld_acquire_u64(&p.flags[first + i]) != epoch) {
                if (globaltimer_ns() - t0 > SP24_WAIT_TIMEOUT_NS) { got = false; break; }
              }
            }
            if (epilogue_bar_any(!got)) { ok = false; break; }
            wsp = p.ws + static_cast<int64_t>(first) * (BN * BM) + c0 * BM + row;
#pragma unroll
            for (int g = 0; g < SK_GRP; ++g)
              if (g < nparts) {
#pragma unroll
                for (int c = 0; c < COLS; ++c) pre[g][c] = __ldcg(wsp + static_cast<int64_t>(g) * (BN * BM) + c * BM);
              }
          }
        }
        if (!mbar_wait(&accf[b], (acc_cnt / NACC) & 1)) ok = false;
        if (SIDE && ok && !mbar_wait(saccf, side_cnt & 1)) ok = false;
        if (epilogue_bar_any(!ok)) { ok = false; break; }
        tc_fence_after();
        const float swr = __ldg(&p.sw[t.b * p.bs_sw + (n >> p.gN_shift)]);
        const float bn = bias_of(p, t.b * p.bs_bias + n);
        if constexpr (BN > 128) {
          // one accumulator: copy this warp's 128 columns to registers and free
          // TMEM at once, so the next tile's MMAs overlap the rest of the epilogue
          uint32_t v[COLS];
#pragma unroll
          for (int c = 0; c < COLS; c += 16) tmem_ld16(lane_base + c0 + c, *reinterpret_cast<uint32_t(*)[16]>(v + c));
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce[b]);  // one arrival per warp
          ++acc_cnt;
          // two passes through the half-size staging buffer: tokens [0,128), then [128,256)
#pragma unroll
          for (int pass = 0; pass < 2; ++pass) {
            if (half == pass) {
#pragma unroll
              for (int j = 0; j < COLS; j += 4)
                scale4_store<false>(scl + c0 + j, swr, v + j, nullptr, bn, out_row + j * 64, 64);
            }
            fence_proxy_async_smem();
            epilogue_bar();
            if (et == 0) {
              tma_store_3d(&tm_y, out_tile, n0, m0 + pass * C::OUT_TOKENS, t.b);
              tma_store_3d(&tm_y, out_tile + C::OUT_TOKENS * 128, n0 + 64, m0 + pass * C::OUT_TOKENS, t.b);
              bulk_commit();
              if (pass == 0) bulk_wait_read_all();
            }
            if (pass == 0) epilogue_bar();
          }
          continue;
        }
        if constexpr (SPLIT || CSPLIT) {
          if (CSPLIT && t.role == 4) {
            // a peer's stages of the cluster's tile: the unscaled fp32 partial
            // goes straight into the leader CTA's shared memory, [peer][col][row],
            // each word counted on the leader's pfull barrier
            const uint32_t peer = cluster_rank() - 1;
            const uint32_t dst = cluster_addr(part, 0) + 4u * (peer * (BN * BM) + c0 * BM + row);
            const uint32_t pbar = cluster_addr(pfull, 0);
#pragma unroll
            for (int c = 0; c < COLS; c += CH) {
              uint32_t v[CH];
              tmem_load_cols<CH / 8>(lane_base + b * BN + c0 + c, v);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < CH; ++j) st_async_b32(dst + 4u * ((c + j) * BM), v[j], pbar);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);  // one arrival per warp
            ++acc_cnt;
            continue;
          }
          if (t.role == 2) {
            // later stages of a tile: publish the unscaled fp32 partial in this
            // CTA's slot, [col][row], for the CTA that holds the tile's start
            float* wpart = p.ws + static_cast<int64_t>(blockIdx.x) * (BN * BM);
#pragma unroll
            for (int c = 0; c < COLS; c += CH) {
              uint32_t v[CH];
              tmem_load_cols<CH / 8>(lane_base + b * BN + c0 + c, v);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < CH; ++j) __stcg(wpart + (c0 + c + j) * BM + row, __uint_as_float(v[j]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);  // one arrival per warp
            ++acc_cnt;
            // the barrier orders every thread's partial before thread 0's
            // releasing store (cumulative at GPU scope): no per-thread fence
            epilogue_bar();
            if (et == 0) st_release_u64(&p.flags[blockIdx.x], epoch);
            continue;
          }
          if (t.role == 1 || t.role == 3) {
            // a tile's first stages complete it: this accumulator, then the
            // partials of the CTAs that hold its later stages, in stage order
            // (a fixed summation order, whatever the arrival order).  Those
            // CTAs start their ranges with these stages and all CTAs are
            // resident, so the waits end.
            float acc[COLS];
#pragma unroll
            for (int c = 0; c < COLS; c += CH) {
              uint32_t v[CH];
              tmem_load_cols<CH / 8>(lane_base + b * BN + c0 + c, v);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < CH; ++j) acc[c + j] = __uint_as_float(v[j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);  // one arrival per warp
            ++acc_cnt;
            if constexpr (CSPLIT) {
              // the peers' partials, in rank order, from this CTA's shared memory
              if (!mbar_wait(pfull, 0)) ok = false;
              if (epilogue_bar_any(!ok)) { ok = false; break; }
              const int peers = static_cast<int>(cluster_nrank()) - 1;
              for (int i = 0; i < peers; ++i) {
                const float* src = part + i * (BN * BM) + c0 * BM + row;
#pragma unroll
                for (int c = 0; c < COLS; ++c) acc[c] += src[c * BM];
              }
            } else {
              // add the partials in CTA order: the gathered group, then the rest
#pragma unroll
              for (int g = 0; g < SK_GRP; ++g)
                if (g < nparts) {
#pragma unroll
                  for (int c = 0; c < COLS; ++c) acc[c] += pre[g][c];
                }
              for (int i = SK_GRP; i < nparts; ++i) {
#pragma unroll
                for (int c = 0; c < COLS; ++c) acc[c] += __ldcg(wsp + static_cast<int64_t>(i) * (BN * BM) + c * BM);
              }
            }
            if (!ok) break;
#pragma unroll
            for (int c = 0; c < COLS; c += 4) {
              const uint32_t a4[4] = {__float_as_uint(acc[c]), __float_as_uint(acc[c + 1]), __float_as_uint(acc[c + 2]),
                                      __float_as_uint(acc[c + 3])};
              scale4_store<false>(scl + c0 + c, swr, a4, nullptr, bn, out_row + (c0 + c) * 64, 64);
            }
            fence_proxy_async_smem();
            epilogue_bar();
            if (et == 0) {
              tma_store_3d(&tm_y, out_tile, n0, m0, t.b);
              tma_store_3d(&tm_y, out_tile + C::OUT_TOKENS * 128, n0 + 64, m0, t.b);
              bulk_commit();
            }
            continue;
          }
        }
#pragma unroll
        for (int c = 0; c < COLS; c += CH) {
          uint32_t v[CH];
          tmem_load_cols<CH / 8>(lane_base + b * BN + c0 + c, v);
          if (SIDE) {
            uint32_t s2[CH];
            tmem_load_cols<CH / 8>(lane_base + NACC * BN + c0 + c, s2);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < CH; j += 4)
              scale4_store<true>(scl + c0 + c + j, swr, v + j, s2 + j, bn, out_row + (c0 + c + j) * 64, 64);
          } else {
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < CH; j += 4)
              scale4_store<false>(scl + c0 + c + j, swr, v + j, nullptr, bn, out_row + (c0 + c + j) * 64, 64);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[b]);  // one arrival per warp
        ++acc_cnt;
        if (SIDE) {
          __syncwarp();
          if (lane == 0) mbar_arrive(sacce);
          ++side_cnt;
        }
      } else {
        // promotion: each K block's partial arrives in its own accumulator buffer;
        // its scales travel in the same pipeline stage (sx[BN], then sw)
        float acc[COLS];
#pragma unroll
        for (int i = 0; i < COLS; ++i) acc[i] = 0.0f;
        const bool per_row_w = p.gN_shift == 0;  // gN = 1: weight scale varies by row
        for (int kt = t.kt0; kt < t.kt1; kt += KS) {
          if (ok && !mbar_wait(&full[e_stage], e_phase)) ok = false;  // scales visible (already complete)
#pragma unroll
          for (int j = 0; j < KS; ++j) {  // K block kt + j: its partial in buffer b, its scales in slot j
            const uint32_t b = acc_cnt % NACC;
            const float* ssl = reinterpret_cast<const float*>(ring + e_stage * C::STAGE + C::SCL_OFF + j * 1024);
            if (ok && !mbar_wait(&accf[b], (acc_cnt / NACC) & 1)) ok = false;
            ok = __all_sync(0xFFFFFFFFu, ok);
            // all of this warp's columns of the partial in one round trip to TMEM
            uint32_t v[COLS];
            if (ok) {
              tc_fence_after();
#pragma unroll
              for (int c = 0; c < COLS; c += CH) tmem_load_cols<CH / 8>(lane_base + b * BN + c0 + c, v + c);
              tmem_ld_wait();
              tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);  // the partial is in registers: the MMA may overwrite its buffer
            if (ok) {
              const float rowf = per_row_w ? ssl[BN + row] : ssl[BN];
#pragma unroll
              for (int i = 0; i < COLS; i += 4) {
                const float4 s4 = *reinterpret_cast<const float4*>(ssl + c0 + i);
                const float2 s01 = __fmul2_rn(make_float2(s4.x, s4.y), make_float2(rowf, rowf));
                const float2 s23 = __fmul2_rn(make_float2(s4.z, s4.w), make_float2(rowf, rowf));
                ffma2(acc[i], acc[i + 1], __uint_as_float(v[i]), __uint_as_float(v[i + 1]), s01.x, s01.y);
                ffma2(acc[i + 2], acc[i + 3], __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]), s23.x, s23.y);
              }
            }
            ++acc_cnt;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[e_stage]);  // this warp is done with the stage's scales
          if (++e_stage == STAGES) { e_stage = 0; e_phase ^= 1; }
        }
        if (epilogue_bar_any(!ok)) { ok = false; break; }
        if (SIDE) {
          if (!mbar_wait(saccf, side_cnt & 1)) ok = false;
          if (epilogue_bar_any(!ok)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < COLS; c += CH) {
            uint32_t s2[CH];
            tmem_load_cols<CH / 8>(lane_base + NACC * BN + c0 + c, s2);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < CH; ++j) acc[c + j] += __uint_as_float(s2[j]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sacce);
          ++side_cnt;
        }
        const float bn = bias_of(p, t.b * p.bs_bias + n);
#pragma unroll
        for (int j = 0; j < COLS; j += 4)
          st_bf16x4(out_row + (c0 + j) * 64, 64, bf16x2_rn(acc[j] + bn, acc[j + 1] + bn),
                    bf16x2_rn(acc[j + 2] + bn, acc[j + 3] + bn));
      }
      // hand the staged tile to the TMA engine: rows past M are clipped by it
      fence_proxy_async_smem();
      epilogue_bar();
      if (et == 0) {
        tma_store_3d(&tm_y, out_tile, n0, m0, t.b);
        tma_store_3d(&tm_y, out_tile + C::OUT_TOKENS * 128, n0 + 64, m0, t.b);
        bulk_commit();
      }
    }
    if (et == 0) bulk_wait_all();
    if (!ok) atomicOr(p.err, DEVERR_TIMEOUT_EPILOGUE);
  }

  pdl_trigger();  // only teardown is left: the next kernel may begin launching
  tc_fence_before();
  if constexpr (CSPLIT)
    cluster_sync();  // no CTA leaves while a peer may still store into its shared memory
  else
    __syncthreads();
  if (SPLIT && threadIdx.x == 0) {
    // count this CTA out (low 20 bits); the launch's last CTA starts the next
    // epoch with a zero count.  Every CTA read the epoch before any CTA got
    // here, so the whole launch used one epoch, and the next launch (after
    // this one is complete) sees the next.  The counter orders no data (the
    // next launch reads it after this grid has completed), so no fence.
    const unsigned long long old = atomicAdd(p.sk_word, 1ull);
    if ((old & 0xFFFFFull) == gridDim.x - 1) atomicExch(p.sk_word, ((old >> 20) + 1) << 20);
  }
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int BN, bool PROMOTE, bool SIDE, bool SPLIT, int KS, bool CSPLIT = false>
sp24_status launch(const DeviceInfo* dev, const CUtensorMap& x, const CUtensorMap& w2, const CUtensorMap& x2,
                   const CUtensorMap& y, const GemmArgs& args, cudaStream_t stream) {
  using C = Cfg<BN, PROMOTE, SIDE, SPLIT, KS, CSPLIT>;
  auto kern = sp24_gemm_kernel<BN, PROMOTE, SIDE, SPLIT, KS, CSPLIT>;
  static std::atomic<bool> attr_done[64];  // per device ordinal; host threads may race to set it (idempotent)
  if (!attr_done[dev->ordinal].load(std::memory_order_acquire)) {
    if (static_cast<size_t>(C::SMEM) > dev->smem_optin) return SP24_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return SP24_ERR_CUDA;
    attr_done[dev->ordinal].store(true, std::memory_order_release);
  }
  if constexpr (CSPLIT) {
    // one cluster of args.cs CTAs per tile (every tile's K range split cs ways)
    const int64_t tiles = static_cast<int64_t>(args.L) * args.m_tiles * args.n_tiles;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(args.cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * args.cs), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, x, w2, x2, y, args) != cudaSuccess) return SP24_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SP24_OK : SP24_ERR_CUDA;
  }
  // stream-K: one CTA per range of stages (at most one per SM); otherwise
  // persistent CTAs over whole tiles
  const int64_t units = SPLIT ? args.sk_units : static_cast<int64_t>(args.L) * args.m_tiles * args.n_tiles;
  const int grid = static_cast<int>(units < dev->sm_count ? units : dev->sm_count);
  if (launch_pdl(kern, dim3(grid), dim3(NUM_THREADS), C::SMEM, stream, x, w2, x2, y, args) != cudaSuccess)
    return SP24_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SP24_OK : SP24_ERR_CUDA;
}

// Sub-tiles per stage for a token tile: small tiles batch more K per stage.
constexpr int ks_for(int bn, bool promote) {
  return promote ? 2 : (bn <= 32 ? 4 : (bn <= 128 ? 2 : 1));
}

template <bool PROMOTE, bool SIDE>
sp24_status launch_bn(int bn, int ks, const DeviceInfo* dev, const CUtensorMap& x, const CUtensorMap& w2,
                      const CUtensorMap& x2, const CUtensorMap& y, const GemmArgs& args, cudaStream_t s) {
  const bool split = args.sk_units > 0;
  const bool csplit = args.cs > 1;
  constexpr bool PLAIN = !PROMOTE && !SIDE;
  switch (bn) {
    case 16:
      if constexpr (!PROMOTE) {
        if (ks == 4) {
          if constexpr (PLAIN) if (split) return launch<16, false, false, true, 4>(dev, x, w2, x2, y, args, s);
          if constexpr (PLAIN) if (csplit) return launch<16, false, false, false, 4, true>(dev, x, w2, x2, y, args, s);
          return launch<16, false, SIDE, false, 4>(dev, x, w2, x2, y, args, s);
        }
      }
      if constexpr (PROMOTE) {
        if (ks == 2) return launch<16, true, SIDE, false, 2>(dev, x, w2, x2, y, args, s);
      }
      return launch<16, PROMOTE, SIDE, false, 1>(dev, x, w2, x2, y, args, s);
    case 32:
      if constexpr (!PROMOTE) {
        if (ks == 4) {
          if constexpr (PLAIN) if (split) return launch<32, false, false, true, 4>(dev, x, w2, x2, y, args, s);
          if constexpr (PLAIN) if (csplit) return launch<32, false, false, false, 4, true>(dev, x, w2, x2, y, args, s);
          return launch<32, false, SIDE, false, 4>(dev, x, w2, x2, y, args, s);
        }
      }
      if constexpr (PROMOTE) {
        if (ks == 2) return launch<32, true, SIDE, false, 2>(dev, x, w2, x2, y, args, s);
      }
      return launch<32, PROMOTE, SIDE, false, 1>(dev, x, w2, x2, y, args, s);
    case 64:
      if constexpr (!PROMOTE) {
        if (ks == 2) {
          if constexpr (PLAIN) if (split) return launch<64, false, false, true, 2>(dev, x, w2, x2, y, args, s);
          if constexpr (PLAIN) if (csplit) return launch<64, false, false, false, 2, true>(dev, x, w2, x2, y, args, s);
          return launch<64, false, SIDE, false, 2>(dev, x, w2, x2, y, args, s);
        }
      }
      if constexpr (PROMOTE) {
        if (ks == 2) return launch<64, true, SIDE, false, 2>(dev, x, w2, x2, y, args, s);
      }
      return launch<64, PROMOTE, SIDE, false, 1>(dev, x, w2, x2, y, args, s);
    case 256:
      if constexpr (PLAIN) return launch<256, false, false, false, 1>(dev, x, w2, x2, y, args, s);
      return SP24_ERR_UNSUPPORTED;
    default:
      if constexpr (!PROMOTE) {
        if (ks == 2) return launch<128, false, SIDE, false, 2>(dev, x, w2, x2, y, args, s);
      }
      if constexpr (PROMOTE) {
        if (ks == 2) return launch<128, true, SIDE, false, 2>(dev, x, w2, x2, y, args, s);
      }
      return launch<128, PROMOTE, SIDE, false, 1>(dev, x, w2, x2, y, args, s);
  }
}

// Token tile: the smallest MMA N that covers M, up to 128; 256 for large M
// when the plain epilogue applies (one accumulator of 256 columns).
int pick_bn(int64_t M, bool plain) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (plain && M > 192) return 256;
  return 128;
}

struct Plan {
  int bn, ks, m_tiles, n_tiles, k_tiles;
  bool streamk;
  int cs;                        // cluster split: CTAs per tile (1 = none)
  int grid;                      // stream-K: CTAs (one range each)
  size_t ws_ctrl, ws_bytes;  // stream-K: control bytes (counter, flags); total with the partials
};

// Bytes of the stream-K control region: the launch counter, then one flag per
// possible CTA (at most one per SM), rounded up to 1 KiB.  It depends on the
// device only, so every shape finds its counter and flags at the same place.
constexpr size_t streamk_ctrl_bytes(int sm_count) {
  return (64 + 8 * static_cast<size_t>(sm_count) + 1023) & ~size_t(1023);
}

// How the tiles' K ranges are dealt out (sp24_set_decomposition): the
// heuristic below, whole tiles only, or stream-K wherever it applies.
std::atomic<int> g_decomposition{SP24_DECOMP_HEURISTIC};

// Stream-K and the cluster split apply to the HBM-bound small-token tiles
// (plain scaling, BN <= 64).  The heuristic models each schedule's time in
// microseconds from the weight bytes (the activations are read from L2 by
// every tile and count in none of them) and constants measured on the
// 152-SM part, and leaves whole tiles only for a gain above 0.1 us:
//  - whole tiles: the busiest CTA streams `rounds` tiles at the rate one SM
//    sustains alone (about 87 GB/s), at best the HBM rate (about 6.5 TB/s);
//  - cluster split, cs = 2 or 4 CTAs per tile, all clusters in one wave: a
//    cs-th of a tile per SM, at best the HBM rate, plus about 1.2 us for the
//    exchange through distributed shared memory (clusters of 3 measured
//    slower than whole tiles: they do not pack the SMs);
//  - stream-K: the HBM rate, plus about 3.5 us for publishing and gathering
//    the partials through L2, plus the completing CTA's read of the partials
//    of a tile's other CTAs (about 150 GB/s).
Plan make_plan(int64_t M, int64_t N, int64_t K, bool promote, bool side, int sm_count, int64_t L) {
  Plan pl;
  pl.bn = pick_bn(M, !promote && !side);
  pl.m_tiles = static_cast<int>((M + pl.bn - 1) / pl.bn);
  pl.n_tiles = static_cast<int>(N / BM);
  pl.k_tiles = static_cast<int>(K / BK);
  pl.ks = ks_for(pl.bn, promote);
  while (pl.ks > 1 && pl.k_tiles % pl.ks != 0) pl.ks /= 2;  // stages hold whole sub-tile groups
  const int64_t tiles = L * pl.m_tiles * pl.n_tiles;
  const int64_t kst = pl.k_tiles / pl.ks;
  pl.streamk = false;
  pl.cs = 1;
  pl.grid = 0;
  pl.ws_ctrl = pl.ws_bytes = 0;
  const int mode = g_decomposition.load(std::memory_order_relaxed);
  if (!promote && !side && pl.bn <= 64 && kst >= 2 && sm_count > 0 && mode != SP24_DECOMP_DATA_PARALLEL) {
    const int cs_max = pl.bn <= 32 ? 4 : 2;  // the leader's shared memory holds 3 (1) peer partials
    auto cs_fits = [&](int cs) { return tiles * cs <= sm_count && kst >= cs; };
    if (mode == SP24_DECOMP_STREAM_K) {
      pl.streamk = true;
    } else if (mode == SP24_DECOMP_CLUSTER_SPLIT) {
      for (int cs = cs_max; cs >= 2 && pl.cs == 1; cs /= 2)
        if (cs_fits(cs)) pl.cs = cs;
    } else {
      const double rounds = static_cast<double>((tiles + sm_count - 1) / sm_count);
      const double tile_bytes = static_cast<double>(pl.k_tiles) * (BM * BK / 2 + BM * BK / 8);
      const double t_hbm = static_cast<double>(tiles) * tile_bytes / 6.5e6;
      const double t_whole = std::max(rounds * tile_bytes / 87e3, t_hbm);
      double best = t_whole - 0.1;
      if (kst >= 4) {
        const double ctas_per_tile = std::min<double>(static_cast<double>(sm_count), static_cast<double>(tiles * kst)) /
                                     static_cast<double>(tiles);
        const double t = t_hbm + 3.5 + (ctas_per_tile - 1.0) * pl.bn * BM * 4 / 150e3;
        if (t < best) {
          best = t;
          pl.streamk = true;
        }
      }
      for (int cs = 2; cs <= cs_max; cs *= 2) {
        if (!cs_fits(cs) || kst < 2 * cs) continue;
        const double t = std::max(tile_bytes / cs / 87e3, t_hbm) + 1.2;
        if (t <= best) {  // on a tie the larger split: more SMs streaming
          best = t;
          pl.cs = cs;
          pl.streamk = false;
        }
      }
    }
  }
  if (pl.streamk) {
    pl.grid = static_cast<int>(std::min<int64_t>(tiles * kst, sm_count));
    pl.ws_ctrl = streamk_ctrl_bytes(sm_count);
    pl.ws_bytes = pl.ws_ctrl + static_cast<size_t>(pl.grid) * pl.bn * BM * sizeof(float);
  }
  return pl;
}

int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

}  // namespace
}  // namespace sp24

extern "C" sp24_status sp24_set_decomposition(int mode) {
  if (mode != SP24_DECOMP_HEURISTIC && mode != SP24_DECOMP_DATA_PARALLEL && mode != SP24_DECOMP_STREAM_K &&
      mode != SP24_DECOMP_CLUSTER_SPLIT)
    return SP24_ERR_INVALID_ARG;
  sp24::g_decomposition.store(mode, std::memory_order_relaxed);
  return SP24_OK;
}

extern "C" int sp24_fp8_gemm_decomposition(int64_t M, int64_t N, int64_t K, int64_t r, int* cluster_size) {
  using namespace sp24;
  if (cluster_size) *cluster_size = 1;
  if (M < 1 || N < BM || N % BM != 0 || K < BK || K % BK != 0 || r < 0) return -1;
  const int sms = current_sm_count();
  if (sms <= 0) return -1;
  if (pair_gemm_applies(M, N, K, true, r)) return SP24_DECOMP_DATA_PARALLEL;
  const Plan pl = make_plan(M, N, K, false, r > 0, sms, 1);
  if (cluster_size) *cluster_size = pl.cs;
  if (pl.streamk) return SP24_DECOMP_STREAM_K;
  return pl.cs > 1 ? SP24_DECOMP_CLUSTER_SPLIT : SP24_DECOMP_DATA_PARALLEL;
}

extern "C" size_t sp24_fp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int64_t r) {
  using namespace sp24;
  if (M < 1 || N < BM || N % BM != 0 || K < BK || K % BK != 0 || r < 0) return 0;
  const int sms = current_sm_count();
  if (sms <= 0) return 0;
  // the workspace depends on the scale granularity only through promotion; size it for the
  // per-tensor-K case, which is the one that can use stream-K
  return make_plan(M, N, K, false, r > 0, sms, 1).ws_bytes;
}

namespace sp24 {
namespace {

// A batch of L problems of one shape: per-problem offsets of every operand
// (bytes for Xq, values and meta; elements for the scales, the bias and Y).
struct Batch {
  int64_t L = 1;
  int64_t x = 0, values = 0, meta = 0, sx = 0, sw = 0, bias = 0, y = 0;
};

sp24_status gemm_impl(const void* Xq, const float* sx, int64_t M, int64_t K, int64_t ldx, int gM, const void* values,
                      const void* meta, const float* sw, int64_t N, int gN, int gK, const void* X2, const void* W2,
                      int64_t r, const void* bias, void* Y, int64_t ldy, const Batch& bt, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!Xq || !sx || !values || !meta || !sw || !Y) return SP24_ERR_INVALID_ARG;
  if (M < 1 || N < 128 || N % 128 != 0 || K < 128 || K % 128 != 0) return SP24_ERR_INVALID_ARG;
  if (M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return SP24_ERR_INVALID_ARG;
  if (ldx < K || ldy < N) return SP24_ERR_INVALID_ARG;
  if ((gM != 1 && gM != 128) || (gN != 1 && gN != 128) || (gK != K && gK != 128)) return SP24_ERR_UNSUPPORTED;
  if (r < 0) return SP24_ERR_INVALID_ARG;
  const bool side = r > 0;
  if (side) {
    if (!X2 || !W2) return SP24_ERR_INVALID_ARG;
    if (r % 16 != 0 || r > 64) return SP24_ERR_UNSUPPORTED;
    if (!aligned16(X2) || !aligned16(W2)) return SP24_ERR_ALIGNMENT;
  }
  if (!aligned16(Xq) || !aligned16(values) || !aligned16(meta) || ldx % 16 != 0) return SP24_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(sx) | reinterpret_cast<uintptr_t>(sw)) % 4 != 0) return SP24_ERR_ALIGNMENT;
  if (!aligned16(Y) || ldy % 8 != 0) return SP24_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(bias) % 2 != 0) return SP24_ERR_ALIGNMENT;
  const DeviceInfo* dev = nullptr;
  sp24_status st = current_device(&dev);
  if (st != SP24_OK) return st;

  const bool promote = (gK == 128 && K != 128);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (bt.L > 1 && (pair_gemm_applies(M, N, K, !promote, r) || (promote && pair_promote_applies(M, N, K, r)))) {
    // problems that fill the GPU on their own: one SM-pair launch each, back
    // to back on the stream (each launch's prologue overlaps the previous tail)
    for (int64_t b = 0; b < bt.L; ++b) {
      const sp24_status e = gemm_impl(
          static_cast<const uint8_t*>(Xq) + b * bt.x, sx + b * bt.sx, M, K, ldx, gM,
          static_cast<const uint8_t*>(values) + b * bt.values, static_cast<const uint8_t*>(meta) + b * bt.meta,
          sw + b * bt.sw, N, gN, gK, X2, W2, r, bias ? static_cast<const uint16_t*>(bias) + b * bt.bias : nullptr,
          static_cast<uint16_t*>(Y) + b * bt.y, ldy, Batch{}, workspace, workspace_bytes, stream);
      if (e != SP24_OK) return e;
    }
    return SP24_OK;
  }
  Plan pl = make_plan(M, N, K, promote, side, dev->sm_count, bt.L);
  if (pl.streamk && (workspace == nullptr || workspace_bytes < pl.ws_bytes || !aligned16(workspace)))
    pl.streamk = false;  // no (or too small a) workspace: whole tiles
  GemmArgs a;
  a.values = static_cast<const uint8_t*>(values);
  a.meta = static_cast<const uint8_t*>(meta);
  a.sx = sx;
  a.sw = sw;
  a.bias = static_cast<const uint16_t*>(bias);
  a.L = static_cast<int>(bt.L);
  a.bs_values = bt.values;
  a.bs_meta = bt.meta;
  a.bs_sx = bt.sx;
  a.bs_sw = bt.sw;
  a.bs_bias = bt.bias;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.ldsx = static_cast<int>((M + gM - 1) / gM);
  a.ldsw = static_cast<int>((N + gN - 1) / gN);
  a.gM_shift = gM == 128 ? 7 : 0;
  a.gN_shift = gN == 128 ? 7 : 0;
  a.m_tiles = pl.m_tiles;
  a.n_tiles = pl.n_tiles;
  a.k_tiles = pl.k_tiles;
  a.side_ksteps = static_cast<int>(r / 16);
  a.kst = pl.k_tiles / pl.ks;
  a.cs = pl.cs;
  a.sk_units = 0;
  a.ws = nullptr;
  a.flags = nullptr;
  a.sk_word = nullptr;
  a.err = dev->err_word;
  if (bt.L * a.m_tiles * a.n_tiles * a.kst >= (int64_t(1) << 31)) return SP24_ERR_UNSUPPORTED;  // 32-bit schedule
  // large token counts with plain scaling: 256 x 256 tiles on SM pairs
  if (pair_gemm_applies(M, N, K, !promote, r))
    return launch_pair_gemm(dev, Xq, ldx, Y, ldy, X2, W2, r, a, s);
  // and with group-wise promotion: 256 x 128 tiles on SM pairs
  if (promote && pair_promote_applies(M, N, K, r)) return launch_pair_promote(dev, Xq, ldx, Y, ldy, a, s);

  const int bn = pl.bn;
  CUtensorMap tm_x, tm_w2, tm_x2, tm_y;
  // [L][M][K] activations and [L][M][N] outputs: a problem's tail rows read
  // zeros and are not stored, whatever its neighbour in the batch holds
  st = make_tmap_3d(&tm_x, Xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, bt.L, ldx, bt.L > 1 ? bt.x : M * ldx, BK, bn,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == SP24_OK)
    st = make_tmap_3d(&tm_y, Y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, bt.L, ldy * 2,
                      (bt.L > 1 ? bt.y : M * ldy) * 2, 64, bn > 128 ? bn / 2 : bn, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st == SP24_OK && side) {
    st = make_tmap_2d(&tm_w2, W2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, r, N, r * 2, 64, BM,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == SP24_OK)
      st = make_tmap_2d(&tm_x2, X2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, r, M, r * 2, 64, bn,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    tm_w2 = tm_x;
    tm_x2 = tm_x;
  }
  if (st != SP24_OK) return st;

  if (pl.streamk) {
    // control words first, at offsets that depend on the device only: the
    // launch counter, whose epoch advances with every launch (on the device,
    // so graph replays advance it too), and one flag per CTA.  A flag an
    // earlier launch left, of any shape, never reads as this launch's, so a
    // workspace zeroed once needs no clearing between calls.  Then one
    // partial tile per CTA.
    a.sk_units = bt.L * a.m_tiles * a.n_tiles * static_cast<int64_t>(a.kst);
    a.sk_word = static_cast<unsigned long long*>(workspace);
    a.flags = a.sk_word + 8;
    a.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.ws_ctrl);
  }
  if (promote)
    return side ? launch_bn<true, true>(bn, pl.ks, dev, tm_x, tm_w2, tm_x2, tm_y, a, s)
                : launch_bn<true, false>(bn, pl.ks, dev, tm_x, tm_w2, tm_x2, tm_y, a, s);
  return side ? launch_bn<false, true>(bn, pl.ks, dev, tm_x, tm_w2, tm_x2, tm_y, a, s)
              : launch_bn<false, false>(bn, pl.ks, dev, tm_x, tm_w2, tm_x2, tm_y, a, s);
}

}  // namespace
}  // namespace sp24

extern "C" sp24_status sp24_fp8_gemm(const void* Xq, const float* sx, int64_t M, int64_t K, int64_t ldx, int gM,
                                     const void* values, const void* meta, const float* sw, int64_t N, int gN,
                                     int gK, const void* X2, const void* W2, int64_t r, const void* bias, void* Y,
                                     int64_t ldy, void* workspace, size_t workspace_bytes, void* stream) {
  return sp24::gemm_impl(Xq, sx, M, K, ldx, gM, values, meta, sw, N, gN, gK, X2, W2, r, bias, Y, ldy, sp24::Batch{},
                         workspace, workspace_bytes, stream);
}

extern "C" sp24_status sp24_fp8_gemm_batched(const void* Xq, const float* sx, int64_t M, int64_t K, int64_t ldx,
                                             int gM, const void* values, const void* meta, const float* sw, int64_t N,
                                             int gN, int gK, const void* bias, void* Y, int64_t ldy, int64_t L,
                                             int64_t stride_x, int64_t stride_sx, int64_t stride_values,
                                             int64_t stride_meta, int64_t stride_sw, int64_t stride_bias,
                                             int64_t stride_y, void* workspace, size_t workspace_bytes,
                                             void* stream) {
  using namespace sp24;
  if (L < 1 || L > (1 << 20)) return SP24_ERR_INVALID_ARG;
  if (M < 1 || N < 128 || K < 128 || ldx < K || ldy < N) return SP24_ERR_INVALID_ARG;
  if (gK != K && gK != 128) return SP24_ERR_UNSUPPORTED;
  const int64_t nsx = (K / gK) * ((M + gM - 1) / gM), nsw = (K / gK) * ((N + gN - 1) / gN);
  if (L > 1) {
    // problems may not overlap: each stride covers at least one problem
    if (stride_x < M * ldx || stride_values < N * K / 2 || stride_meta < N * K / 8 || stride_sx < nsx ||
        stride_sw < nsw || stride_y < M * ldy || (bias && stride_bias < N))
      return SP24_ERR_INVALID_ARG;
    if (stride_x % 16 != 0 || stride_values % 16 != 0 || stride_meta % 16 != 0 || (stride_y * 2) % 16 != 0)
      return SP24_ERR_ALIGNMENT;
  }
  Batch bt;
  bt.L = L;
  bt.x = stride_x;
  bt.values = stride_values;
  bt.meta = stride_meta;
  bt.sx = stride_sx;
  bt.sw = stride_sw;
  bt.bias = stride_bias;
  bt.y = stride_y;
  return gemm_impl(Xq, sx, M, K, ldx, gM, values, meta, sw, N, gN, gK, nullptr, nullptr, 0, bias, Y, ldy, bt,
                   workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free GEMM entry point.
//
// Some callers own their device-memory budget outright and must not allocate
// once they are running: serving loops that plan every buffer at start-up,
// or code hosted inside a framework whose allocator this library cannot
// reach.  For them the stream-K scratch of sp24_fp8_gemm comes from the fixed
// array below instead of a caller-provided workspace.  The array lives in
// this library's device image, so every GPU that loads the library holds it
// (kFixedScratchBytes) until the process exits, and all calls on a device
// share it.
namespace sp24 {
namespace {

constexpr size_t kFixedScratchBytes = size_t(8) << 20;  // 8 MiB per device
static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

// The largest stream-K scratch is the control region plus one 64-token
// partial tile per CTA, with at most one CTA per SM (make_plan).  Every part
// with up to kFixedScratchMaxSMs SMs (the 152-SM GB300 among them) fits the
// array at every shape, so the refusal in the entry point is a guard for
// larger parts; a change of tile sizes that breaks this bound fails here.
constexpr int kFixedScratchMaxSMs = 240;
static_assert(streamk_ctrl_bytes(kFixedScratchMaxSMs) +
                      static_cast<size_t>(kFixedScratchMaxSMs) * 64 * BM * sizeof(float) <=
                  kFixedScratchBytes,
              "the fixed scratch holds every stream-K plan of a part with up to kFixedScratchMaxSMs SMs");

// Device address of the scratch array in the current device's context.  In
// host code the array's name is only a host-side handle; the runtime maps it
// to the device copy.  The lookup runs on every call (cheap once the
// library's device image is loaded), so a context that was reset and created
// again never receives a stale address.
sp24_status fixed_scratch_address(void** out) {
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_fixed_scratch) != cudaSuccess || addr == nullptr) return SP24_ERR_CUDA;
  *out = addr;
  return SP24_OK;
}

}  // namespace
}  // namespace sp24

extern "C" sp24_status sp24_fp8_gemm_fixed_scratch(const void* Xq, const float* sx, int64_t M, int64_t K, int64_t ldx,
                                                   int gM, const void* values, const void* meta, const float* sw,
                                                   int64_t N, int gN, int gK, const void* X2, const void* W2,
                                                   int64_t r, const void* bias, void* Y, int64_t ldy, void* stream) {
  using namespace sp24;
  // scratch this shape needs (stream-K partials, flags and counter); more than the
  // fixed array holds is refused rather than silently run another way
  if (sp24_fp8_gemm_workspace_size(M, N, K, r) > kFixedScratchBytes) return SP24_ERR_WORKSPACE;
  void* scratch = nullptr;
  const sp24_status st = fixed_scratch_address(&scratch);
  if (st != SP24_OK) return st;
  // The scratch starts zeroed (a static device array) and the stream-K
  // control words keep it consistent from call to call.
  return sp24_fp8_gemm(Xq, sx, M, K, ldx, gM, values, meta, sw, N, gN, gK, X2, W2, r, bias, Y, ldy, scratch,
                       kFixedScratchBytes, stream);
}
