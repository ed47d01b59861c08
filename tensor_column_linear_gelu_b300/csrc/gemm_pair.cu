// gemm_pair.cu -- tcgen05 / TMEM tensor-core GEMM on CTA pairs, fed by TMA,
// for bf16 calls with many tokens (prefill-shaped).
//
//   column-parallel:  Y_i = act(X . W_i^T + b_i) for every shard i in one launch;
//                     the shard index is a group of N-tiles, shard i's tiles
//                     write its column block.  Fused epilogue: bias, erf-GELU,
//                     or SwiGLU (the packed gate/up shard puts the 128 gate
//                     columns and the matching 128 up columns of an output
//                     group into one 256-wide tile).
//   row-parallel:     Y = sum_i X_i . W_i^T + b.  The K loop walks shard 0's
//                     k-blocks, then shard 1's, ... into ONE TMEM accumulator:
//                     that accumulator is the all-reduce's sum.  The bias is
//                     added once, in the epilogue.
// ("Understanding Tensor Parallelism for Multi-GPU LLM Serving", "How Tensor
// Parallelism Works Under the Hood"; "Tensor parallel serving",
// "Column-parallel and row-parallel layers, paired".)
//
// Structure: clusters of two CTAs (a pair), one cluster per 256 x 256 output
// tile in the grid; the clusters that run steal the tiles of those that have
// not started (cluster launch control), so each runs many tiles.  One MMA
// (tcgen05.mma.cta_group::2, M=256, N=256, K=16) covers the pair's tile: the
// even CTA issues it, each CTA holds 128 of the tile's rows
// of A (tokens) and 128 of its rows of B (weights) in shared memory, and
// each CTA's TMEM holds the accumulator of its 128 token rows.  Per SM this
// halves the weight bytes loaded and read per FLOP compared with a 128 x 256
// tile on one SM.
//   warp 0      TMA producer (both CTAs): this CTA's A and B halves of each
//               64-wide k-block into a 6-stage ring; completion is counted on
//               the even CTA's barrier, which expects both halves.  The even
//               CTA's producer also asks for the pair's next tile when it
//               starts a tile.
//   warp 1      TMEM allocation (both CTAs, collectively) and, in the even
//               CTA, the single thread that issues the MMAs, committing each
//               stage back to both producers and each finished tile to both
//               epilogues (multicast commits).
//   warps 2-5   epilogue (both CTAs): tcgen05.ld of this CTA's accumulator
//               rows (one TMEM lane = one token row per thread), bias /
//               activation in fp32, one rounding, stores; then an arrive on
//               the even CTA's accumulator-free barrier.
// Every mbarrier wait is bounded (sync.cuh); a wait that gives up records the
// failure in the device error word, raises the CTA's abort flag, and the
// roles unwind.  Every thread of both CTAs reaches the closing cluster
// barrier and the collective TMEM release whatever happened.
//
// Summation order of an output element: k-blocks in increasing k (then, on
// the row side, shard by shard), 4 MMAs of K=16 per k-block.  It does not
// depend on N or tp, so column-parallel outputs are bit-identical to tp = 1.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sync.cuh"
#include "tc_ptx.cuh"

namespace tpla {
namespace {

constexpr int PM = 256;             // tokens per pair tile (MMA M)
constexpr int HM = PM / 2;          // tokens per CTA (TMEM lanes)
constexpr int PN = 256;             // output columns per tile (MMA N)
constexpr int HN = PN / 2;          // weight rows of B per CTA
constexpr int BK = 64;              // k per stage: 64 bf16 = 128 bytes = one swizzle span
constexpr int UMMA_K = 16;
constexpr int STAGES = 6;
constexpr int A_BYTES = HM * BK * 2;  // 16 KB
constexpr int B_BYTES = HN * BK * 2;  // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int ACC_BUFS = 2;
constexpr int TMEM_COLS = 512;      // ACC_BUFS x PN fp32 columns
constexpr int THREADS = 192;
constexpr int EPI_WARP0 = 2;
constexpr int CLC_SLOTS = 4;        // answers of the tile scheduler in flight
// readers of each answer: both producers, the MMA thread, 8 epilogue warps
constexpr int CLC_READERS = 2 + 1 + 8;
constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_BUFS + 1 + 2 * CLC_SLOTS;
constexpr int SMEM_BYTES =
    1024 /*align slack*/ + STAGES * STAGE_BYTES + CLC_SLOTS * 16 + NUM_BARS * 8 + 16;
constexpr int64_t G = TP_GATE_UP_GROUP;
static_assert(2 * G == PN, "a SwiGLU tile holds one gate/up group");
static_assert(SMEM_BYTES <= 232448, "dynamic shared memory per CTA");

// One GEMM of a launch.  A launch runs one problem, or two independent ones
// (the attention projections: QKV and O) whose tiles share the grid, so the
// partial last wave of each is filled by the other's tiles.
struct PairProblem {
  int a_map, b_map;  // first tensor map of A (column: X; row: X_i) and of B (W_i) in tm[]
  const float* bias[TP_MAX_TP];
  void* Y;
  int64_t y_extent;  // elements of Y this problem may write (checked builds)
  int64_t ldy, y_shard_stride;
  int64_t M, ns, n_out;
  int tp, row, act, ydt;
  int m_tiles, n_tiles_per_shard, n_tiles, num_tiles;
  int kb_per_shard, kb_total;
  int tile0;         // first tile of this problem in the launch's tile sequence
};
constexpr int kPairMaxProblems = 2;
// a column problem needs 1 + tp maps, a row problem 2 tp: a column and a row
// problem together at most 1 + 3 TP_MAX_TP
constexpr int kPairMaxMaps = 1 + 3 * TP_MAX_TP;

struct PairParams {
  CUtensorMap tm[kPairMaxMaps];  // boxes {64, 128}
  PairProblem prob[kPairMaxProblems];
  int nprob, num_tiles, nmaps;
  unsigned int* err;
};

__device__ __forceinline__ int valid_count(int64_t limit, int64_t n) {
  const int64_t rem = limit - n;
  return rem <= 0 ? 0 : (rem >= 32 ? 32 : (int)rem);
}

struct TileCoord {
  int shard;   // column: shard of this tile; row: unused
  int64_t m0;  // first token of the pair's tile
  int64_t n0;  // first row of W_i (column) or first output column (row)
};

// The problem a tile of the launch belongs to, and its index inside it.
__device__ __forceinline__ const PairProblem& problem_of(const PairParams& p, int tile, int& lt) {
  const int q = (p.nprob > 1 && tile >= p.prob[1].tile0) ? 1 : 0;
  lt = tile - p.prob[q].tile0;
  return p.prob[q];
}

// Tiles are numbered M-fastest within groups of up to GROUP_M m-tiles, and the
// groups are swept one after the other: the pairs running at the same time
// share the weight tiles they stream, and a group's activations (2048 tokens)
// stay in L2 while the weights pass through.  Tiles start in this order
// (clusters launch, and are cancelled, in grid order), so the pairs that
// share a weight tile start it within a few microseconds of each other, and
// the weights are read from DRAM little more than once per group.  Odd groups sweep the
// n-tiles backwards, starting with the weight tiles the previous group read
// last.
constexpr int GROUP_M = 8;
__device__ __forceinline__ TileCoord tile_coord(const PairProblem& p, int tile) {
  const int per_group = GROUP_M * p.n_tiles;
  const int g = tile / per_group;
  const int m_first = g * GROUP_M;
  const int gm = min(GROUP_M, p.m_tiles - m_first);  // m-tiles in this group
  const int t = tile - g * per_group;
  const int mt = m_first + t % gm;
  const int nt = (g & 1) ? p.n_tiles - 1 - t / gm : t / gm;
  TileCoord c;
  c.m0 = (int64_t)mt * PM;
  if (p.row) {
    c.shard = 0;
    c.n0 = (int64_t)nt * PN;
  } else {
    c.shard = nt / p.n_tiles_per_shard;
    c.n0 = (int64_t)(nt % p.n_tiles_per_shard) * PN;
  }
  return c;
}

// The pair's tile after its j-th: answer j of the scheduler (slot j mod
// CLC_SLOTS, that slot's (j / CLC_SLOTS)-th use).  Each reader waits for the
// answer in its own CTA, reads it, and arrives on the even CTA's cempty, so
// the slot is asked again only once all CLC_READERS have read it.  A warp
// calls it with every lane (whole_warp) and one arrive.  Returns the tile, -1
// when the scheduler had nothing left, -2 when the wait gave up.
__device__ __forceinline__ int next_tile(const uint8_t* clc_resp, uint64_t* cfull,
                                         uint32_t cempty_lead, int j, const volatile int* abort,
                                         bool whole_warp) {
  const int s = j % CLC_SLOTS;
  bool ok = mbar_wait_bounded(smem_u32(&cfull[s]), (uint32_t)(j / CLC_SLOTS) & 1u, kWaitLimitNs,
                              abort);
  if (whole_warp) ok = __all_sync(0xffffffffu, ok);
  if (!ok) return -2;
  const int x = clc_cancelled_first_x(smem_u32(clc_resp + s * 16));
  if (whole_warp) __syncwarp();
  if (!whole_warp || (threadIdx.x & 31) == 0) {
    fence_proxy_async_smem();  // the read above is ordered before the slot's next answer
    mbar_arrive_cluster(cempty_lead + (uint32_t)(s * 8));
  }
  return x < 0 ? -1 : (x >> 1);
}

__global__ void __launch_bounds__(THREADS, 1) gemm_pair_kernel(const __grid_constant__ PairParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* clc_resp = sB + STAGES * B_BYTES;  // CLC_SLOTS answers of 16 bytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(clc_resp + CLC_SLOTS * 16);
  uint64_t* full = bars;                 // even CTA's are used: both halves land there
  uint64_t* empty = bars + STAGES;       // each CTA's own: its producer waits on it
  uint64_t* tfull = bars + 2 * STAGES;   // each CTA's own: its epilogue waits on it
  uint64_t* tempty = tfull + ACC_BUFS;   // even CTA's: both epilogues arrive
  uint64_t* drain = tempty + ACC_BUFS;
  uint64_t* cfull = drain + 1;           // each CTA's own: an answer has landed here
  uint64_t* cempty = cfull + CLC_SLOTS;  // even CTA's: every reader of an answer arrives
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + NUM_BARS) + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: even CTA of the pair, 1: odd
  const bool lead = rank == 0;
  const int own_tile = blockIdx.x >> 1;  // this cluster's tile; later ones are stolen
  const uint32_t cempty_lead = dsmem_addr(smem_u32(&cempty[0]), 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < ACC_BUFS; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), 8);  // one arrive per epilogue warp of both CTAs
    }
    mbar_init(smem_u32(drain), 1);
    for (int s = 0; s < CLC_SLOTS; ++s) {
      mbar_init(smem_u32(&cfull[s]), 1);  // armed by this CTA's producer (16 bytes)
      mbar_init(smem_u32(&cempty[s]), CLC_READERS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.nmaps; ++i) prefetch_tmap(&p.tm[i]);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), TMEM_COLS);
  // Both CTAs' barriers are initialised and the TMEM address is known before
  // any copy, MMA or remote arrive targets them.
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int pending = -1;  // use of the answer slot armed here and not yet read
    int tile = own_tile;
    for (int j = 0; tile >= 0 && ok; ++j) {
      const int s = j % CLC_SLOTS;
      if (lead) {
        // ask for the next tile now: the answer is back long before this
        // tile's loads are issued
        if (!mbar_wait_bounded(smem_u32(&cempty[s]), ((uint32_t)(j / CLC_SLOTS) & 1u) ^ 1u,
                               kWaitLimitNs, abort_flag)) {
          report_error(p.err, kErrTimeoutProducer);
          *abort_flag = 1;
          break;
        }
        fence_proxy_async_smem();
        clc_try_cancel_all(smem_u32(clc_resp + s * 16), smem_u32(&cfull[s]));
      }
      mbar_arrive_expect_tx(smem_u32(&cfull[s]), 16);
      pending = j;
      int lt;
      const PairProblem& P = problem_of(p, tile, lt);
      const TileCoord c = tile_coord(P, lt);
      // The K loop as (shard, k-block in shard): a row problem walks its tp
      // shards, a column problem its one shard's k-blocks.  This one thread
      // issues every copy of the pair's half, two per k-block, and a k-block
      // takes the MMAs about 0.28 us: a division per k-block to find the
      // shard made the row launches 8-14 % slower.
      const int nsh = P.row ? P.tp : 1;
      const int nkk = P.row ? P.kb_per_shard : P.kb_total;
      const int ya = (int)(c.m0 + (int64_t)rank * HM);
      const int yb = (int)(c.n0 + (int64_t)rank * HN);
      for (int si = 0; si < nsh && ok; ++si) {
        const CUtensorMap* ma = &p.tm[P.a_map + (P.row ? si : 0)];
        const CUtensorMap* mb = &p.tm[P.b_map + (P.row ? si : c.shard)];
        for (int kk = 0; kk < nkk; ++kk) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, kWaitLimitNs, abort_flag)) {
            report_error(p.err, kErrTimeoutProducer);
            *abort_flag = 1;
            ok = false;
            break;
          }
          const uint32_t fb_own = smem_u32(&full[stage]);
          const uint32_t fb = dsmem_addr(fb_own, 0);  // the even CTA's barrier
          if (lead) mbar_arrive_expect_tx(fb_own, 2 * STAGE_BYTES);
          tma_load_2d_pair(smem_u32(sA + stage * A_BYTES), ma, kk * BK, ya, fb);
          tma_load_2d_pair(smem_u32(sB + stage * B_BYTES), mb, kk * BK, yb, fb);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) break;
      tile = next_tile(clc_resp, cfull, cempty_lead, j, abort_flag, false);
      pending = -1;
      if (tile == -2) {
        report_error(p.err, kErrTimeoutProducer);
        *abort_flag = 1;
        break;
      }
    }
    // An answer asked for and not read (after a failure) lands before this
    // CTA can leave: wait for it without regard to the abort flag.
    if (pending >= 0)
      (void)mbar_wait_bounded(smem_u32(&cfull[pending % CLC_SLOTS]),
                              (uint32_t)(pending / CLC_SLOTS) & 1u, kWaitLimitNs);
    // Every copy issued here is consumed by an MMA (the even CTA issues them
    // for the same tile sequence), and this CTA's epilogue waits for the
    // commit that follows the last one; the closing cluster barrier follows.
  } else if (warp == 1 && lane == 0 && lead) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t IDESC = idesc_bf16_f32(PM, PN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    int tile = own_tile;
    for (int j = 0; tile >= 0 && ok; ++j) {
      int lt;
      const PairProblem& P = problem_of(p, tile, lt);
      if (!mbar_wait_bounded(smem_u32(&tempty[acc]), acc_phase ^ 1u, kWaitLimitNs, abort_flag)) {
        report_error(p.err, kErrTimeoutMma);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * PN);
      for (int kb = 0; kb < P.kb_total; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, kWaitLimitNs, abort_flag)) {
          report_error(p.err, kErrTimeoutMma);
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t adesc = sdesc_sw128(smem_u32(sA + stage * A_BYTES));
        const uint64_t bdesc = sdesc_sw128(smem_u32(sB + stage * B_BYTES));
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k) {
          // advance the start address by k * 32 bytes inside the swizzle span
          mma_bf16_pair(d_tmem, adesc + (uint64_t)(k * 2), bdesc + (uint64_t)(k * 2), IDESC,
                        (kb > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit_pair_mc(smem_u32(&empty[stage]), 0x3);  // both producers may refill
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      mma_commit_pair_mc(smem_u32(&tfull[acc]), 0x3);  // both epilogues may read
      if (++acc == ACC_BUFS) {
        acc = 0;
        acc_phase ^= 1u;
      }
      tile = next_tile(clc_resp, cfull, cempty_lead, j, abort_flag, false);
      if (tile == -2) {
        report_error(p.err, kErrTimeoutMma);
        *abort_flag = 1;
        break;
      }
    }
    // every MMA this thread issued has completed before TMEM is released
    mma_commit_pair(smem_u32(drain));
    if (!mbar_wait_bounded(smem_u32(drain), 0, kWaitLimitNs)) report_error(p.err, kErrTimeoutDrain);
  } else if (warp >= EPI_WARP0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;             // TMEM lane quadrant this warp may access
    const int row_in_tile = (int)rank * HM + q * 32 + lane;
    const uint32_t tempty_lead = dsmem_addr(smem_u32(&tempty[0]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    int tile = own_tile;
    for (int j = 0; tile >= 0; ++j) {
      // all lanes wait, then agree: tcgen05.ld below is warp-collective, so
      // the warp must never split on a timeout
      bool ok = mbar_wait_bounded(smem_u32(&tfull[acc]), acc_phase, kWaitLimitNs, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) report_error(p.err, kErrTimeoutEpilogue);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      int lt;
      const PairProblem& P = problem_of(p, tile, lt);
      const bool swiglu = (!P.row && P.act == TP_ACT_SWIGLU);
      const TileCoord c = tile_coord(P, lt);
      const int64_t m = c.m0 + row_in_tile;
      const bool row_ok = m < P.M;
      const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * PN);
      if (swiglu) {
        // tile = one packed group: gate columns [0,128), up columns [128,256)
        const int64_t out0 = (c.n0 / (2 * G)) * G;   // first output of the group (shard-local)
        const int64_t base = (int64_t)c.shard * P.y_shard_stride + m * P.ldy;
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          float g[32], u[32];
          tmem_ld32(trow + ch * 32, g);
          tmem_ld32(trow + G + ch * 32, u);
#pragma unroll
          for (int j = 0; j < 32; ++j) g[j] = act_silu(g[j]) * u[j];
          const int64_t n = out0 + ch * 32;
          const int valid = valid_count(P.ns, n);
          if (row_ok && valid > 0 && TP_CHECK(p.err, base + n + valid <= P.y_extent))
            store_row32(P.Y, P.ydt, base, n, valid, g);
        }
      } else {
        const int64_t limit = P.row ? P.n_out : P.ns;
        const int64_t base = (P.row ? 0 : (int64_t)c.shard * P.y_shard_stride) + m * P.ldy;
        const float* bias = P.row ? P.bias[0] : P.bias[c.shard];
#pragma unroll 1
        for (int ch = 0; ch < PN / 32; ++ch) {
          float v[32];
          tmem_ld32(trow + ch * 32, v);
          const int64_t n = c.n0 + ch * 32;
          const int valid = valid_count(limit, n);
          if (bias) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < valid) v[j] += __ldg(bias + n + j);
          }
          if (!P.row && P.act == TP_ACT_GELU_ERF) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = act_gelu_erf(v[j]);
          }
          if (row_ok && valid > 0 && TP_CHECK(p.err, base + n + valid <= P.y_extent))
            store_row32(P.Y, P.ydt, base, n, valid, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_lead + (uint32_t)(acc * 8));
      if (++acc == ACC_BUFS) {
        acc = 0;
        acc_phase ^= 1u;
      }
      tile = next_tile(clc_resp, cfull, cempty_lead, j, abort_flag, true);
      if (tile == -2) {
        if (lane == 0) report_error(p.err, kErrTimeoutEpilogue);
        *abort_flag = 1;
        break;
      }
    }
  }

  __syncthreads();
  // No CTA of the pair leaves (or frees TMEM) while the other may still arrive
  // on its barriers or while MMAs may still write its TMEM: the even CTA's
  // MMA thread has waited for its last MMA before this barrier.
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

}  // namespace

namespace {

// Fill problem q of the launch from a validated LinearProblem, encoding its
// tensor maps from tm[*nmaps] on.
bool fill_problem(const LinearProblem& p, PairParams& gp, int q, int* nmaps) {
  PairProblem& P = gp.prob[q];
  const int64_t es = 2;
  if (*nmaps + (p.row ? 2 * p.tp : 1 + p.tp) > kPairMaxMaps) return false;
  P.a_map = *nmaps;
  if (p.row) {
    for (int i = 0; i < p.tp; ++i) {
      const void* xi = static_cast<const char*>(p.X) + (int64_t)i * p.x_shard_off * es;
      if (!make_tma_map_bf16(&gp.tm[(*nmaps)++], xi, (uint64_t)p.K, (uint64_t)p.M,
                             (uint64_t)(p.ldx * es), HM))
        return false;
    }
  } else if (!make_tma_map_bf16(&gp.tm[(*nmaps)++], p.X, (uint64_t)p.K, (uint64_t)p.M,
                                (uint64_t)(p.ldx * es), HM)) {
    return false;
  }
  P.b_map = *nmaps;
  for (int i = 0; i < p.tp; ++i)
    if (!make_tma_map_bf16(&gp.tm[(*nmaps)++], p.W[i], (uint64_t)p.K, (uint64_t)p.w_rows,
                           (uint64_t)(p.K * es), HN))
      return false;
  for (int i = 0; i < TP_MAX_TP; ++i) P.bias[i] = p.bias[i];
  P.Y = p.Y;
  P.ldy = p.ldy;
  P.y_extent = output_extent(p);
  P.y_shard_stride = p.y_shard_stride;
  P.M = p.M;
  P.ns = p.ns;
  P.n_out = p.n_out;
  P.tp = p.tp;
  P.row = p.row ? 1 : 0;
  P.act = p.act;
  P.ydt = p.ydt;
  P.m_tiles = (int)((p.M + PM - 1) / PM);
  P.kb_per_shard = (int)((p.K + BK - 1) / BK);
  if (p.row) {
    P.n_tiles_per_shard = (int)((p.n_out + PN - 1) / PN);
    P.n_tiles = P.n_tiles_per_shard;
    P.kb_total = P.kb_per_shard * p.tp;
  } else {
    P.n_tiles_per_shard = (int)((p.w_rows + PN - 1) / PN);
    P.n_tiles = P.n_tiles_per_shard * p.tp;
    P.kb_total = P.kb_per_shard;
  }
  const int64_t tiles = (int64_t)P.m_tiles * P.n_tiles;
  if (tiles > INT32_MAX / 2) return false;
  P.num_tiles = (int)tiles;
  return true;
}

tp_status finish_launch(PairParams& gp, Launch* L) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return TP_ERR_CUDA;
  // One cluster per tile: the clusters that run take over the tiles of those
  // not yet started, in grid order.
  L->kernel = reinterpret_cast<const void*>(gemm_pair_kernel);
  L->grid = dim3((unsigned)(2 * std::max(gp.num_tiles, 1)));
  L->block = dim3(THREADS);
  L->smem = (size_t)SMEM_BYTES;
  L->cluster = 2;
  L->set_params(gp);
  return TP_OK;
}

}  // namespace

tp_status prepare_gemm_pair(const LinearProblem& p, Launch* L) {
  PairParams gp{};
  gp.err = device_error_word();
  if (!gp.err) return TP_ERR_CUDA;
  int nmaps = 0;
  if (!fill_problem(p, gp, 0, &nmaps)) return TP_ERR_CUDA;
  gp.nprob = 1;
  gp.nmaps = nmaps;
  gp.prob[0].tile0 = 0;
  gp.num_tiles = gp.prob[0].num_tiles;
  return finish_launch(gp, L);
}

tp_status prepare_gemm_pair2(const LinearProblem& a, const LinearProblem& b, Launch* L) {
  PairParams gp{};
  gp.err = device_error_word();
  if (!gp.err) return TP_ERR_CUDA;
  int nmaps = 0;
  if (!fill_problem(a, gp, 0, &nmaps) || !fill_problem(b, gp, 1, &nmaps)) return TP_ERR_CUDA;
  gp.nprob = 2;
  gp.nmaps = nmaps;
  gp.prob[0].tile0 = 0;
  gp.prob[1].tile0 = gp.prob[0].num_tiles;
  gp.num_tiles = gp.prob[0].num_tiles + gp.prob[1].num_tiles;
  return finish_launch(gp, L);
}

}  // namespace tpla
