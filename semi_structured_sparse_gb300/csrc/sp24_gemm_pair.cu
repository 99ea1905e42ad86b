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
// The kernel is launched with programmatic stream serialisation: its
// prologue (barriers, TMEM, descriptor prefetch) overlaps the previous
// kernel's tail, and pdl_wait() precedes every global-memory access.
#include <cuda_bf16.h>
#include "sp24_gemm_common.cuh"

namespace sp24 {
namespace {

constexpr int PN = 256;                        // tokens per pair tile (MMA N)
constexpr int HALF_N = PN / 2;                 // activation rows each CTA loads
constexpr int KS = 2;                          // K blocks per stage
constexpr int P_B = HALF_N * BK;               // 16 KB of activations per CTA per K block
constexpr int P_A_OFF = 0;                     // KS values tiles (contiguous in the tiled storage)
constexpr int P_META_OFF = KS * A_STAGE;       // KS metadata tiles
constexpr int P_B_OFF = KS * (A_STAGE + META_STAGE);
constexpr int P_STAGE = P_B_OFF + KS * P_B;    // bytes each CTA receives per stage
constexpr int P_OUT_TOKENS = 64;               // tokens per staged store pass
constexpr int P_OUT_BYTES = P_OUT_TOKENS * BM * 2;
constexpr int P_SCALE_BYTES = 4 * PN;
constexpr int P_FIXED = 1024 + P_OUT_BYTES + P_SCALE_BYTES + BAR_BYTES;
constexpr int P_STAGES_FIT = (SMEM_LIMIT - P_FIXED) / P_STAGE;
constexpr int P_STAGES = P_STAGES_FIT < META_SLOTS / KS ? P_STAGES_FIT : META_SLOTS / KS;
constexpr int P_SMEM = P_FIXED + P_STAGES * P_STAGE;
constexpr int P_COLS = PN / 2;                 // accumulator columns per epilogue warp
constexpr int CHUNK = 32;                      // token chunk: warp half h holds chunks h, h + 2, ...
constexpr int NPASS = PN / P_OUT_TOKENS;
constexpr int VROWS = A_STAGE / 128;           // a values tile is 64 rows of 128 B
constexpr int MROWS = META_STAGE / 128;        // a metadata tile is 16 rows of 128 B
static_assert(P_B_OFF % 1024 == 0 && P_STAGE % 1024 == 0, "1024-byte swizzle alignment");
static_assert(P_STAGES >= 3 && P_STAGES <= MAX_STAGES, "pipeline depth");
static_assert(PN <= META_COL0, "TMEM columns");
static_assert(P_OUT_TOKENS == 2 * CHUNK, "each pass takes one chunk from each warp half");
static_assert(P_STAGES * P_STAGE >= PN * BM * 2, "the ring holds a whole output tile");

__global__ void __launch_bounds__(NUM_THREADS, 1)
    sp24_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_m, const __grid_constant__ CUtensorMap tm_y,
                          const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base by pointer arithmetic on the shared array, so that
  // accesses through it compile to shared-memory instructions
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = sm;
  uint8_t* out_tile = sm + P_STAGES * P_STAGE;                     // [2 channel halves][64 tokens][64] bf16
  float* scl = reinterpret_cast<float*>(out_tile + P_OUT_BYTES);  // token scales of the tile [PN]
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_tile + P_OUT_BYTES + P_SCALE_BYTES);
  uint64_t* full = bars;                  // [P_STAGES] leader: both CTAs' loads -> MMA
  uint64_t* empty = bars + MAX_STAGES;    // [P_STAGES] each CTA: MMA done with the stage -> its loads
  uint64_t* accf = bars + 2 * MAX_STAGES; // each CTA: accumulator complete -> its epilogue
  uint64_t* acce = accf + 1;              // leader: both epilogues drained the accumulator -> MMA
  uint64_t* drain = acce + 1;             // leader: every MMA finished (before TMEM is freed)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(num_clusters_x());
  const int num_units = p.m_tiles * p.n_tiles;
  const int k_stages = (p.k_tiles + KS - 1) / KS;
  if (threadIdx.x == 0) {
    for (int i = 0; i < P_STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(accf, 1);
    mbar_init(acce, 2 * EPI_WARPS);  // one arrival per epilogue warp of each CTA
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == MMA_WARP + 1 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_m);
    tma_prefetch_desc(&tm_y);
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
      for (int ks = 0; ks < k_stages; ++ks, ++flat) {
        if (flat % PRODUCERS != warp) continue;
        const uint32_t stage = static_cast<uint32_t>(flat % P_STAGES);
        const uint32_t phase = static_cast<uint32_t>((flat / P_STAGES) & 1);
        const bool got = mbar_wait(&empty[stage], phase ^ 1);
        if (!__all_sync(0xFFFFFFFFu, got)) { ok = false; break; }
        if (lane == 0) {
          // Always KS blocks: with an odd block count the last stage's second
          // block reads the next weight tile's rows (or zero fill past the end)
          // and K coordinates past K (zero fill); the MMA skips it.
          const int kt = ks * KS;
          const uint32_t fb = full0 + 8u * stage;
          uint8_t* st = ring + stage * P_STAGE;
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * P_STAGE);  // both CTAs' bytes
          tma_load_2d_pair(st + P_A_OFF, &tm_v, fb, 0, vrow + kt * VROWS);
          tma_load_2d_pair(st + P_META_OFF, &tm_m, fb, 0, mrow + kt * MROWS);
#pragma unroll
          for (int j = 0; j < KS; ++j) tma_load_2d_pair(st + P_B_OFF + j * P_B, &tm_x, fb, (kt + j) * BK, m0);
        }
      }
    }
    if (lane == 0) {
      if (!ok) atomicOr(p.err, DEVERR_TIMEOUT_PRODUCER);
      // Before leaving: the MMA has released every stage this warp filled (so its
      // copies have landed and nothing writes this CTA's shared memory later).
      // Only the last use of a slot may be waited on.
      const int64_t fmax = flat - 1;
      for (int64_t f = fmax; f >= 0 && f > fmax - P_STAGES; --f) {
        if (f % PRODUCERS != warp) continue;
        (void)mbar_wait(&empty[f % P_STAGES], static_cast<uint32_t>((f / P_STAGES) & 1));
      }
    }
  } else if (warp == MMA_WARP) {
    // ----------------------------------------------------------- MMA issuer
    if (leader && lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3(2 * BM, PN, true);
      constexpr uint64_t STAGE_DESC = P_STAGE >> 4;
      const uint32_t ring_u32 = smem_u32(ring);
      const uint64_t a_desc0 = smem_desc(ring_u32 + P_A_OFF, 16, 512, SWZ_64B);
      const uint64_t m_desc0 = smem_desc(ring_u32 + P_META_OFF, 128, 128, SWZ_NONE);
      const uint64_t b_desc0 = smem_desc(ring_u32 + P_B_OFF, 16, 1024, SWZ_128B);
      uint32_t stage = 0, phase = 0, meta_ctr = 0, acc_cnt = 0;
      bool ok = true;
      for (int u = pair; u < num_units && ok; u += npairs) {
        if (!mbar_wait(acce, (acc_cnt & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        for (int ks = 0; ks < k_stages; ++ks) {
          if (!mbar_wait(&full[stage], phase)) { ok = false; break; }
          tc_fence_after();
          const uint64_t off = stage * STAGE_DESC;
          const int nsub = min(KS, p.k_tiles - ks * KS);
#pragma unroll
          for (int j = 0; j < KS; ++j) {
            if (j < nsub) {
              const uint32_t mcol = tbase + META_COL0 + 4 * (meta_ctr & (META_SLOTS - 1));
              ++meta_ctr;
              tmem_cp_128x128b_pair(mcol, m_desc0 + off + j * (META_STAGE >> 4));
              const uint64_t aj = a_desc0 + off + j * (A_STAGE >> 4);
              const uint64_t bj = b_desc0 + off + j * (P_B >> 4);
              mma_sp_e4m3_pair(tbase, aj, bj, mcol, idesc, (ks != 0 || j != 0) ? 1u : 0u);
              mma_sp_e4m3_pair(tbase, aj + 2, bj + 4, mcol + 2, idesc, 1u);  // +32 B of A, +64 B of B
            }
          }
          mma_commit_pair(&empty[stage], 3);
          if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit_pair(accf, 3);
        ++acc_cnt;
      }
      if (!ok) atomicOr(p.err, DEVERR_TIMEOUT_MMA);
      mma_commit_pair(drain, 1);  // every MMA issued must finish before TMEM is freed
      (void)mbar_wait(drain, 0);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int ew = warp - EPI_WARP0;              // 0..7
    const int q = warp & 3;                       // TMEM lane quadrant this warp may access
    const int half = ew >> 2;                     // token chunks half, half + 2, half + 4, half + 6
    const int row = 32 * q + lane;                // weight row within this CTA's 128
    const int et = threadIdx.x - 32 * EPI_WARP0;  // 0..EPI_THREADS-1
    const uint32_t lane_base = tbase + (static_cast<uint32_t>(32 * q) << 16);
    const uint32_t acce_leader = cluster_addr(acce, 0);
    uint32_t acc_cnt = 0;
    bool ok = true;
    for (int u = pair; u < num_units && ok; u += npairs) {
      const bool last = u + npairs >= num_units;  // this CTA's final tile: the ring is free afterwards
      const int n0 = (2 * (u % p.n_tiles) + static_cast<int>(rank)) * BM;  // this CTA's channels
      const int m0 = (u / p.n_tiles) * PN;                                  // the tile's tokens
      const int n = n0 + row;
      if (et == 0) bulk_wait_read_all();  // the previous tile's stores have read the staging buffer
      {
        const int m = m0 + et;
        scl[et] = m < p.M ? __ldg(&p.sx[m >> p.gM_shift]) : 0.0f;
      }
      // loaded before the accumulator is waited on, so that nothing is
      // outstanding when the accumulator is released (a release arrive waits)
      const float swr = __ldg(&p.sw[n >> p.gN_shift]);
      if (!mbar_wait(accf, acc_cnt & 1)) ok = false;
      if (epilogue_bar_any(!ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t v[P_COLS];  // chunk i of this warp: tokens CHUNK * (half + 2 i) + [0, CHUNK)
#pragma unroll
      for (int i = 0; i < P_COLS / CHUNK; ++i) {
        const uint32_t col = lane_base + CHUNK * (half + 2 * i);
        tmem_ld16(col, *reinterpret_cast<uint32_t(*)[16]>(v + CHUNK * i));
        tmem_ld16(col + 16, *reinterpret_cast<uint32_t(*)[16]>(v + CHUNK * i + 16));
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce_leader);  // the next tile's MMAs may overwrite TMEM
      ++acc_cnt;
      if (last) {
        // whole tile through the idle ring: [channel half][256 tokens][64 channels] bf16
        uint16_t* ring_row = reinterpret_cast<uint16_t*>(ring) + (row >> 6) * (PN * 64) + (row & 63);
#pragma unroll
        for (int i = 0; i < P_COLS / CHUNK; ++i) {
          const int t0 = CHUNK * (half + 2 * i);
#pragma unroll
          for (int j = 0; j < CHUNK; j += 4)
            scale4_store<false>(scl + t0 + j, swr, v + CHUNK * i + j, nullptr, ring_row + (t0 + j) * 64, 64);
        }
        fence_proxy_async_smem();
        epilogue_bar();
        if (et == 0) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int t = 0; t < PN; t += P_OUT_TOKENS)
              tma_store_2d(&tm_y, ring + c * (PN * 128) + t * 128, n0 + 64 * c, m0 + t);
          bulk_commit();
        }
      } else {
        // four passes of 64 tokens through the staging buffer; in pass s every
        // warp converts its chunk s (tokens 64 s + 32 half + [0, 32))
        uint16_t* out_row = reinterpret_cast<uint16_t*>(out_tile) + (row >> 6) * (P_OUT_TOKENS * 64) + (row & 63);
#pragma unroll
        for (int s = 0; s < NPASS; ++s) {
          const int t0 = P_OUT_TOKENS * s + CHUNK * half;
#pragma unroll
          for (int j = 0; j < CHUNK; j += 4)
            scale4_store<false>(scl + t0 + j, swr, v + CHUNK * s + j, nullptr, out_row + (CHUNK * half + j) * 64, 64);
          fence_proxy_async_smem();
          epilogue_bar();
          if (et == 0) {
            tma_store_2d(&tm_y, out_tile, n0, m0 + P_OUT_TOKENS * s);
            tma_store_2d(&tm_y, out_tile + P_OUT_TOKENS * 128, n0 + 64, m0 + P_OUT_TOKENS * s);
            bulk_commit();
            if (s < NPASS - 1) bulk_wait_read_all();
          }
          if (s < NPASS - 1) epilogue_bar();
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

bool pair_gemm_applies(int64_t M, int64_t N, int64_t K, bool plain) {
  // 256-token tiles pay off from a little under one full tile; TMA row
  // coordinates of the tiled weight views must fit in int32
  return plain && M > 192 && N % (2 * BM) == 0 && (N / 256) * (K + BK) < (int64_t(1) << 31);
}

sp24_status launch_pair_gemm(const DeviceInfo* dev, const void* Xq, int64_t ldx, const void* Y, int64_t ldy,
                             const GemmArgs& args_in, cudaStream_t stream) {
  GemmArgs a = args_in;
  const int64_t M = a.M, N = a.N, K = a.K;
  a.m_tiles = static_cast<int>((M + PN - 1) / PN);
  a.n_tiles = static_cast<int>(N / (2 * BM));
  a.k_tiles = static_cast<int>(K / BK);
  a.splits = 1;
  a.kt_per_split = a.k_tiles;
  CUtensorMap tm_x, tm_v, tm_m, tm_y;
  sp24_status st = make_tmap_2d(&tm_x, Xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, ldx, BK, HALF_N,
                                CU_TENSOR_MAP_SWIZZLE_128B);
  // tiled weight storage as 128-byte rows: a values tile is 64 rows, a metadata tile 16
  if (st == SP24_OK)
    st = make_tmap_2d(&tm_v, a.values, CU_TENSOR_MAP_DATA_TYPE_UINT8, 128, N * K / 256, 128, 128, KS * VROWS,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st == SP24_OK)
    st = make_tmap_2d(&tm_m, a.meta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 128, N * K / 1024, 128, 128, KS * MROWS,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st == SP24_OK)
    st = make_tmap_2d(&tm_y, Y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, ldy * 2, 64, P_OUT_TOKENS,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != SP24_OK) return st;

  auto kern = sp24_gemm_pair_kernel;
  static int max_pairs[64] = {};  // per device: co-resident pairs (0 = not yet known)
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
  cfg.dynamicSmemBytes = P_SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_pairs[d] == 0) {
    if (static_cast<size_t>(P_SMEM) > dev->smem_optin) return SP24_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM) != cudaSuccess)
      return SP24_ERR_CUDA;
    cfg.gridDim = dim3(2 * (dev->sm_count / 2), 1, 1);
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess || active < 1) return SP24_ERR_CUDA;
    max_pairs[d] = active;
  }
  const int units = a.m_tiles * a.n_tiles;
  const int pairs = units < max_pairs[d] ? units : max_pairs[d];
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, kern, tm_x, tm_v, tm_m, tm_y, a) != cudaSuccess) return SP24_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SP24_OK : SP24_ERR_CUDA;
}

}  // namespace sp24
