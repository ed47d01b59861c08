// skinny.cu -- tcgen05 / TMEM kernel for decode-shaped bf16 calls: a handful
// of tokens (up to kSkinnyMaxTokens) against a large weight.
//
// With few tokens a linear layer reads every weight byte once and does about
// M FLOPs per byte, so it is bound by HBM bandwidth: each device streams its
// own slice of the weights ("What is tensor parallelism?", "Why it helps when
// serving").  Three measured facts shape the kernel:
//   * a tcgen05.mma of M=128, K=16 occupies the tensor core for about the same
//     time whatever N is, so the weights must be the N operand: one MMA then
//     consumes up to 256 weight rows x 16 k (8 KB).  The tokens are the
//     128-row A operand; only the first M rows are loaded, the other rows of
//     the A tile (whatever shared memory holds) only produce TMEM lanes that
//     nothing reads;
//   * TMA streaming reaches the HBM roofline with 128-byte-wide boxes, so a
//     deep ring of (X box, weight rows) stages per SM is enough;
//   * every SM must stream about the same number of bytes, or the SMs that
//     finish early leave bandwidth unused.
//
//   column-parallel:  Y_i = act(X . W_i^T + b_i).  CTA b of a persistent grid
//                     owns the output features [b*F/grid, (b+1)*F/grid) in
//                     units of 8 (features numbered shard-major).  The range
//                     is cut into pieces that stay inside one shard (and, for
//                     SwiGLU, one gate/up group), and consecutive pieces are
//                     packed at 16-row slots into one B tile of up to 512
//                     weight rows (two MMAs of N <= 256 per k-step), so a CTA
//                     normally runs a single K loop with every stage full.  Every
//                     output accumulates over all of K in one TMEM column,
//                     so its summation order depends on K only and sharded
//                     results are bit-identical to tp = 1.
//                     With fewer than SK_SPLIT_ROWS weight rows per CTA the
//                     walk is bound by the fixed cost of each MMA instead:
//                     then clusters of cs CTAs take 256-row tiles (features
//                     [t*256, (t+1)*256), SwiGLU 128 gate + 128 up) and split
//                     the K loop, and their partials are summed in rank order
//                     as on the row side below.  The choice depends on F, K,
//                     M and the SM count, not on the shards, so tp = 1 makes
//                     the same one and the results stay bit-identical.
//                     SwiGLU: a piece's gate rows sit at its slot among the
//                     tile's first R rows and its up rows at the same slot
//                     among the next R (R = slot rows of the tile, <= 256);
//                     the thread that owns a token reads gate column slot+j
//                     and up column R+slot+j of the accumulator.
//   row-parallel:     Y = sum_i X_i . W_i^T + b.  The outputs are cut into
//                     tiles of 256; each tile belongs to a thread-block
//                     cluster of cs CTAs that split the K loop (shard 0's
//                     k-blocks, then shard 1's, ...) into cs contiguous parts.
//                     Each CTA's partial sum goes TMEM -> its shared memory;
//                     after a cluster barrier CTA r adds the cs partials of
//                     its slice of the tile in rank order (distributed shared
//                     memory loads), adds the bias once and stores.  With
//                     cs = tp each CTA holds exactly one shard's partial and
//                     the cluster reduction is the all-reduce's sum.
// ("Understanding Tensor Parallelism for Multi-GPU LLM Serving", "How Tensor
// Parallelism Works Under the Hood"; "Tensor parallel serving",
// "Column-parallel and row-parallel layers, paired".)
//
// Roles (192 threads, 704 in FP8 mode; one CTA per SM):
//   warp 0      TMA producer: per k-block one X box {64, xrows} (lane 0) and
//               the tile's weight rows as 64-row and 16-row boxes, one box
//               per lane: a single thread issuing many small boxes cannot
//               keep the TMA unit busy.
//   warp 1      TMEM allocation (512 columns: one accumulator of up to 512
//               fp32 columns, or two when they fit) and the single thread
//               issuing tcgen05.mma (M=128, N<=256, K=16), committing each
//               stage back to the producer and each finished tile to the
//               epilogue.
//   warps 2-5   epilogue: tcgen05.ld (one TMEM lane = one token per thread),
//               bias / activation in fp32, one rounding, row stores; on the
//               row side the partial goes to shared memory for the cluster
//               reduction.
//   warps 6-21  FP8 mode only: the converters (below).
//
// FP8 mode (e4m3 weight codes + one fp32 scale per weight row; used above
// the token count of the FP8 kernel in decode_fp8.cu, which widens the codes
// into tensor memory instead of shared memory).  The codes
// are streamed at one byte per weight -- half the bytes of bf16, which is the
// point for a call bound by weight bytes -- and widened on chip:
//   * the producer loads the same rows as in bf16 mode, SK_KPR k-blocks of
//     codes wide (128 bytes), into a ring of raw stages (no swizzle);
//   * sixteen converter warps (two groups taking alternate k-blocks) turn
//     each k-block of a raw stage into a bf16 B tile laid out
//     exactly as a 128-byte-swizzled TMA load would have left it (16-byte
//     chunk c of row r at chunk c ^ (r mod 8)), fence the writes for the
//     async proxy and hand the buffer to the MMA thread.  The widening is
//     exact (every e4m3 value is a bf16 value), so the MMA computes x . q in
//     fp32 as the bf16 path computes x . w;
//   * the epilogue multiplies each output's accumulator by its weight row's
//     scale (gate and up rows each by their own) before the bias and the
//     activation.  On the row side each CTA's k-range lies inside one shard
//     (clusters of tp x j CTAs), so its partial is scaled by that shard's row
//     scales before the cluster sum.
// Three rings: X boxes (released by the MMA's commit), raw code stages
// (released by the converters as soon as they are read, so that most of the
// raw ring is always in flight from HBM) and two bf16 B-tile buffers between
// the converters and the MMA thread.  A B tile holds at most 256 rows (one
// MMA), which keeps the bf16 buffers small and the raw ring deep.
//
// Every mbarrier wait is bounded (sync.cuh); a wait that gives up records the
// failure in the device error word and that role stops issuing work.  Every
// thread of every CTA still reaches both cluster barriers, so a failure can
// never leave a peer CTA waiting.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "decode_tiles.cuh"
#include "internal.h"
#include "sync.cuh"
#include "tc_ptx.cuh"

namespace tpla {
namespace {

using namespace decode;

// This kernel's tile loop: the shared one, with a column tile's K loop
// narrowed to the CTA's k-blocks [skb0, skb1) (all of K unless clusters
// split K).
#undef SK_FOR_EACH_TILE
#define SK_FOR_EACH_TILE(tl, ...)                                     \
  do {                                                                \
    if (p.row) {                                                      \
      const Tile tl = row_tile(p, rank);                              \
      __VA_ARGS__                                                     \
    } else {                                                          \
      for (int64_t f_ = f0; f_ < f1;) {                               \
        Tile t_ = column_tile(p, f_, f1);                             \
        t_.kb0 = skb0;                                                \
        t_.kb1 = skb1;                                                \
        const Tile tl = t_;                                           \
        __VA_ARGS__                                                   \
      }                                                               \
    }                                                                 \
  } while (0)

constexpr int SK_THREADS = 192;
constexpr int SK_EPI_WARP0 = 2;
constexpr int SK_CONV_WARP0 = 6;            // FP8 mode: first converter warp
constexpr int SK_CONV_WARPS = 16;
// Two converter groups take alternate k-blocks, each into its own bf16
// buffer, so that two conversions are in progress at any time.
constexpr int SK_CONV_GROUPS = 2;
constexpr int SK_GROUP_WARPS = SK_CONV_WARPS / SK_CONV_GROUPS;
constexpr int SK_GROUP_THREADS = 32 * SK_GROUP_WARPS;
// a converter thread's rows advance by SK_GROUP_THREADS / 4 per chunk, a
// multiple of 8: its swizzle phase (row mod 8) never changes
static_assert((SK_GROUP_THREADS / 4) % 8 == 0, "converter row stride");
constexpr int SK_THREADS_F8 = SK_THREADS + 32 * SK_CONV_WARPS;
constexpr int SK_BK = 64;                   // k per stage: one 128-byte swizzle span
constexpr int SK_UMMA_K = 16;
constexpr int SK_ROW_BYTES = SK_BK * 2;     // 128 bytes per staged bf16 row
// FP8 mode: a raw stage holds SK_KPR k-blocks of each tile row, so that
// every TMA row request moves SK_KPR x 64 contiguous bytes of codes
constexpr int SK_KPR = 2;
static_assert(SK_KPR == 1 || SK_KPR == 2 || SK_KPR == 4, "k-blocks per raw stage");
constexpr int SK_RAW_ROW_BYTES = SK_BK * SK_KPR;  // bytes per staged row of codes
constexpr int SK_CSTAGES = 2;               // FP8 mode: bf16 B-tile buffers, one per group
constexpr int SK_MAX_CSTAGES = 4;
static_assert(SK_CSTAGES == SK_CONV_GROUPS, "k-block n uses buffer n mod 2, converted by group n mod 2");
constexpr int SK_A_BYTES = 128 * SK_ROW_BYTES;  // the A tile one MMA reads (128 rows)
constexpr int SK_MAX_STAGES = 16;
constexpr int SK_ACC_BUFS = 2;              // accumulator buffers, when two fit in TMEM
constexpr int SK_TMEM_COLS = 512;
constexpr int SK_MAX_CLUSTER = kSkinnyMaxCluster;
constexpr int SK_RED_PITCH = SK_BN + 4;     // floats per token row of a reduction buffer
constexpr int SK_NUM_BARS = 4 * SK_MAX_STAGES + 2 * SK_ACC_BUFS + 1 + 2 * SK_MAX_CSTAGES;
constexpr int SK_BAR_BYTES = SK_NUM_BARS * 8 + 16;
constexpr int SK_SMEM_MAX = 232448;         // dynamic shared memory per CTA (227 KB)
// Column side: below this many weight rows per CTA the feature walk is bound
// by the tensor core's fixed time per MMA (about 140 cycles, whatever N):
// the 8-token QKV projection (80 rows a CTA) took 0.43 us a k-block, 73 us
// for 168 MB.  Such calls give each cluster of cs CTAs a 256-row tile and
// split its K loop instead (partials summed in rank order, as on the row
// side), for up to SK_SPLIT_MAX_TOKENS tokens (the partial-sum buffer sits
// beside the ring), with at least SK_SPLIT_MIN_KB k-blocks per CTA: short
// K loops are not MMA-bound, and there the clusters' fixed costs lose (the
// [16, 512] x 2048 GELU up projection, 8 k-blocks, went from 22 to 60 us
// split 8 ways).  The choice depends on the total feature count, K, M and
// the SM count only, so sharded results stay bit-identical to tp = 1.
constexpr int SK_SPLIT_ROWS = 128;
constexpr int SK_SPLIT_MAX_TOKENS = 32;
constexpr int SK_SPLIT_MIN_KB = 32;

struct SkinnyParams {
  CUtensorMap tmX[TP_MAX_TP];    // column: [0] = X; row: X_i.  Box {64, xrows}.
  CUtensorMap tmW16[TP_MAX_TP];  // W_i, box {64, 16} (FP8 mode: 64 codes x 16 rows)
  CUtensorMap tmW64[TP_MAX_TP];  // W_i, box {64, 64}
  const float* bias[TP_MAX_TP];
  const float* wscale[TP_MAX_TP];  // FP8 mode: scale of each row of W_i
  void* Y;
  unsigned int* err;
  int64_t ldy;
  int64_t y_extent;              // elements of Y this call may write (checked builds)
  int64_t fo[TP_MAX_TP + 1];     // column: shard i owns features [fo[i], fo[i+1])
  int64_t yoff[TP_MAX_TP];       // column: element offset of shard i's outputs in Y
  int64_t M, feat_total;         // feat_total: column fo[tp]; row n_out
  int tp, row, act, ydt;
  int xrows, x_stage_bytes, stages;
  int w_stage_bytes;             // weight rows of a B tile x 128 bytes
  int raw_stage_bytes;           // FP8 mode: weight rows of a B tile x 64 bytes
  int cstages;                   // FP8 mode: bf16 B-tile buffers
  int xstages;                   // FP8 mode: X ring depth (the raw ring has `stages`)
  int tile_cap;                  // column: features (SwiGLU) or rows per tile
  int acc_stride, acc_bufs;      // TMEM columns per accumulator buffer, buffers
  int kb_per_shard, kb_total;
  int cs;                        // CTAs per cluster splitting K (row side, column K split)
  int csplit;                    // column side: clusters of cs CTAs split each tile's K loop
  int ring_bytes;                // shared memory below the barriers (checked builds)
  int red_off, red_bytes;        // column K split: the partial-sum buffer in shared memory
};

template <bool F8>
__global__ void __launch_bounds__(F8 ? SK_THREADS_F8 : SK_THREADS, 1)
    skinny_kernel(const __grid_constant__ SkinnyParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // bf16 mode: S X stages, S weight stages (one ring).  FP8 mode: XS X
  // stages, S raw (e4m3) stages, cstages bf16 B-tile buffers (three rings).
  // All 1024-byte aligned.
  const int S = p.stages;
  const int XS = F8 ? p.xstages : S;
  const int WB = F8 ? p.cstages : S;                       // bf16 B-tile buffers
  uint8_t* sX = smem;
  uint8_t* sR = smem + (size_t)XS * p.x_stage_bytes;       // FP8 mode only
  uint8_t* sW = sR + (F8 ? (size_t)S * p.raw_stage_bytes : 0);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sW + (size_t)WB * p.w_stage_bytes);
  uint64_t* full = bars;                       // X (bf16: X + weights) landed
  uint64_t* empty = bars + SK_MAX_STAGES;      // X stage consumed by the MMAs
  uint64_t* rfull = bars + 2 * SK_MAX_STAGES;  // FP8: codes landed
  uint64_t* rempty = bars + 3 * SK_MAX_STAGES; // FP8: codes read by the converters
  uint64_t* tfull = bars + 4 * SK_MAX_STAGES;
  uint64_t* tempty = tfull + SK_ACC_BUFS;
  uint64_t* drain = tempty + SK_ACC_BUFS;
  uint64_t* cfull = drain + 1;                 // FP8: bf16 buffer converted
  uint64_t* cempty = cfull + SK_MAX_CSTAGES;   // FP8: bf16 buffer consumed by the MMAs
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + SK_NUM_BARS);
  // Row side: after the K loop the ring is reused as this CTA's reduction
  // buffer red[token][SK_RED_PITCH] (fp32).
  float* red = reinterpret_cast<float*>(smem + p.red_off);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool swiglu = (!p.row && p.act == TP_ACT_SWIGLU);
  const int rank = (p.row || p.csplit) ? (int)cluster_ctarank() : 0;
  // row side, FP8 mode: the shard this CTA's k-range lies in
  const int rshard = p.row ? (int)((int64_t)rank * p.tp / p.cs) : 0;
  // The next kernel may start its prologue now.  The producer waits for the
  // kernels before this one before its first load (every stage carries X);
  // everything that writes Y comes after its loads.
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < XS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    if (F8) {
      for (int s = 0; s < S; ++s) {
        mbar_init(smem_u32(&rfull[s]), 1);
        mbar_init(smem_u32(&rempty[s]), SK_CONV_WARPS);  // one arrive per converter warp
      }
    }
    for (int a = 0; a < p.acc_bufs; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), 4);  // one arrive per epilogue warp
    }
    mbar_init(smem_u32(drain), 1);
    if (F8) {
      for (int c = 0; c < p.cstages; ++c) {
        mbar_init(smem_u32(&cfull[c]), SK_GROUP_WARPS);  // one arrive per warp of its group
        mbar_init(smem_u32(&cempty[c]), 1);
      }
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    const int nx = p.row ? p.tp : 1;
    for (int i = 0; i < nx; ++i) prefetch_tmap(&p.tmX[i]);
    for (int i = 0; i < p.tp; ++i) {
      prefetch_tmap(&p.tmW16[i]);
      prefetch_tmap(&p.tmW64[i]);
    }
  }
  if (warp == 1) tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), SK_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int64_t f0 = 0, f1 = 0;
  if (p.csplit)
    column_split_range_of(p, (int64_t)blockIdx.x, f0, f1);
  else if (!p.row)
    column_range(p, f0, f1);
  int skb0 = 0, skb1 = p.kb_total;  // column side: this CTA's k-blocks
  if (p.csplit) split_kb_range(p, rank, skb0, skb1);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp issues: lane 0 waits for the stage(s), arms the barriers
    // and loads the X box; lane 1 + b loads weight box b of the tile.  Issuing
    // the boxes from many lanes keeps the TMA unit fed.  FP8 mode: the X box
    // goes to the X ring, the codes to the raw ring, each with its barriers.
    int stage = 0;      // X ring (bf16 mode: the one ring)
    uint32_t phase = 0;
    int rs = 0;         // FP8: raw ring
    uint32_t rphase = 0;
    bool ok = true;
    // X is re-read by every SM; the weights are streamed once.
    const uint64_t pol_x = l2_policy_evict_last();
    const uint64_t pol_w = l2_policy_evict_first();
    // X may be the output of the kernel before this one (programmatic
    // dependent launch): bf16 mode issues the weight boxes of the first S
    // stages at once and defers their X boxes (lane 0) until pdl_wait, so
    // the weight stream starts while the previous kernel finishes.  FP8 mode
    // waits first.
    bool waited = F8;
    if constexpr (F8) pdl_wait();
    int nd = 0;  // deferred X boxes (lane 0): stage, k-block, shard
    int d_stage[SK_MAX_STAGES], d_kk[SK_MAX_STAGES], d_sh[SK_MAX_STAGES];
    auto flush_x = [&]() {
      if (lane == 0) {
        pdl_wait();
        for (int i = 0; i < nd; ++i)
          tma_load_2d_hint(smem_u32(sX + (size_t)d_stage[i] * p.x_stage_bytes), &p.tmX[d_sh[i]],
                           d_kk[i] * SK_BK, 0, smem_u32(&full[d_stage[i]]), pol_x);
      }
      nd = 0;
      waited = true;
      __syncwarp();
    };
    SK_FOR_EACH_TILE(tl, {
      if (ok) {
        int piece = 0, half = 0, r = 0, h = 0;
        const bool has_box = lane > 0 && tile_box(tl, swiglu, lane - 1, piece, half, r, h);
        int64_t wrow = 0;     // first weight row of this lane's box in its shard buffer
        uint32_t woff = 0;    // its offset in the stage's B tile
        int wshard = 0;
        constexpr int pitch = F8 ? SK_RAW_ROW_BYTES : SK_ROW_BYTES;  // bytes per loaded row
        if (has_box) {
          const Piece& pc = tl.pc[piece];
          wrow = (swiglu ? (pc.loc / G) * 2 * G + pc.loc % G + half * G : pc.loc) + r;
          woff = (uint32_t)(pc.slot + half * tl.rows + r) * pitch;
          wshard = pc.shard;
        }
        const bool mine =
            has_box && TP_CHECK(p.err, woff + (uint32_t)h * pitch <=
                                           (uint32_t)(F8 ? p.raw_stage_bytes : p.w_stage_bytes));
        uint32_t wbytes = 0;  // weight (code) bytes of one stage
        if (lane == 0) {
          for (int b = 0; b < tl.boxes; ++b) {
            int pi, hf, rr, hh;
            if (tile_box(tl, swiglu, b, pi, hf, rr, hh)) wbytes += (uint32_t)hh * pitch;
          }
        }
        if constexpr (F8) {
          // one raw stage per SK_KPR k-blocks (fewer at the end of the range:
          // a box reaching past the shard's K reads zeros that nobody uses),
          // then the X boxes of those k-blocks, one per X stage
          for (int kb = tl.kb0; kb < tl.kb1 && ok; kb += SK_KPR) {
            const int nsub = tl.kb1 - kb < SK_KPR ? tl.kb1 - kb : SK_KPR;
            const int rsh = p.row ? kb / p.kb_per_shard : 0;
            const int kk = p.row ? kb - rsh * p.kb_per_shard : kb;
            bool got = true;
            if (lane == 0) got = mbar_wait_bounded(smem_u32(&rempty[rs]), rphase ^ 1u);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
              if (lane == 0) report_error(p.err, kErrTimeoutProducer);
              ok = false;
              break;
            }
            const uint32_t wb = smem_u32(&rfull[rs]);
            if (lane == 0) {
              mbar_arrive_expect_tx(wb, wbytes);
            } else if (mine) {
              const int sh = p.row ? rsh : wshard;
              const CUtensorMap* map = (h == 64) ? &p.tmW64[sh] : &p.tmW16[sh];
              tma_load_2d_hint(smem_u32(sR + (size_t)rs * p.raw_stage_bytes) + woff, map,
                               kk * SK_BK, (int)wrow, wb, pol_w);
            }
            __syncwarp();
            if (++rs == S) {
              rs = 0;
              rphase ^= 1u;
            }
            for (int j = 0; j < nsub; ++j) {
              bool gx = true;
              if (lane == 0) gx = mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u);
              gx = __shfl_sync(0xffffffffu, gx, 0);
              if (!gx) {
                if (lane == 0) report_error(p.err, kErrTimeoutProducer);
                ok = false;
                break;
              }
              if (lane == 0) {
                const uint32_t fb = smem_u32(&full[stage]);
                mbar_arrive_expect_tx(fb, (uint32_t)p.x_stage_bytes);
                tma_load_2d_hint(smem_u32(sX + (size_t)stage * p.x_stage_bytes), &p.tmX[rsh],
                                 (kk + j) * SK_BK, 0, fb, pol_x);
              }
              __syncwarp();
              if (++stage == XS) {
                stage = 0;
                phase ^= 1u;
              }
            }
          }
        } else {
          // row side: shard rsh and k-block kk inside it, advanced with kb
          int rsh = p.row ? tl.kb0 / p.kb_per_shard : 0;
          int kk = p.row ? tl.kb0 - rsh * p.kb_per_shard : tl.kb0;
          for (int kb = tl.kb0; kb < tl.kb1; ++kb, ++kk) {
            if (p.row && kk == p.kb_per_shard) {
              kk = 0;
              ++rsh;
            }
            if (!waited && nd == S) flush_x();  // stage reuse needs the deferred X boxes
            bool got = true;
            if (lane == 0) got = mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
              if (lane == 0) report_error(p.err, kErrTimeoutProducer);
              ok = false;
              break;
            }
            const uint32_t fb = smem_u32(&full[stage]);
            if (lane == 0) {
              mbar_arrive_expect_tx(fb, (uint32_t)p.x_stage_bytes + wbytes);
              if (waited) {
                tma_load_2d_hint(smem_u32(sX + (size_t)stage * p.x_stage_bytes), &p.tmX[rsh],
                                 kk * SK_BK, 0, fb, pol_x);
              } else if (TP_CHECK(p.err, nd < SK_MAX_STAGES)) {
                d_stage[nd] = stage;
                d_kk[nd] = kk;
                d_sh[nd] = rsh;
              }
            } else if (mine) {
              const int sh = p.row ? rsh : wshard;
              const CUtensorMap* map = (h == 64) ? &p.tmW64[sh] : &p.tmW16[sh];
              tma_load_2d_hint(smem_u32(sW + (size_t)stage * p.w_stage_bytes) + woff, map,
                               kk * SK_BK, (int)wrow, fb, pol_w);
            }
            if (!waited) ++nd;
            __syncwarp();
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    });
    if (!waited) flush_x();  // fewer stages than the ring holds
    // Every copy issued here is consumed by the MMA thread (same tile
    // sequence); the epilogue waits for the commit that follows the last one.
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    int cst = 0;            // FP8 mode: bf16 buffer of this k-block
    uint32_t cphase = 0;
    bool ok = true;
    SK_FOR_EACH_TILE(tl, {
      if (ok && !mbar_wait_bounded(smem_u32(&tempty[acc]), acc_phase ^ 1u)) {
        report_error(p.err, kErrTimeoutMma);
        ok = false;
      }
      if (ok) {
        tc_fence_after();
        const int nrows = swiglu ? 2 * tl.rows : tl.rows;  // gate rows, then up rows
        const int n0 = nrows < SK_BN ? nrows : SK_BN;        // first MMA's N
        const int n1 = nrows - n0;                           // second MMA's N (or 0)
        const uint32_t idesc0 = idesc_bf16_f32(128, n0);
        const uint32_t idesc1 = idesc_bf16_f32(128, n1 > 0 ? n1 : 16);
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * p.acc_stride);
        if (!TP_CHECK(p.err, nrows * SK_ROW_BYTES <= p.w_stage_bytes &&
                                 acc * p.acc_stride + nrows <= SK_TMEM_COLS))
          ok = false;
        for (int kb = tl.kb0; ok && kb < tl.kb1; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase) ||
              (F8 && !mbar_wait_bounded(smem_u32(&cfull[cst]), cphase))) {
            report_error(p.err, kErrTimeoutMma);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_sw128(smem_u32(sX + (size_t)stage * p.x_stage_bytes));
          const uint32_t wbase = smem_u32(sW + (size_t)(F8 ? cst : stage) * p.w_stage_bytes);
          const uint64_t bdesc0 = sdesc_sw128(wbase);
          const uint64_t bdesc1 = sdesc_sw128(wbase + SK_BN * SK_ROW_BYTES);
#pragma unroll
          for (int k = 0; k < SK_BK / SK_UMMA_K; ++k) {
            // advance the start address by k * 32 bytes inside the swizzle span;
            // B rows [0, 256) feed accumulator columns [0, 256), rows [256, ..)
            // columns [256, ..)
            const uint32_t accum = (kb > tl.kb0 || k > 0) ? 1u : 0u;
            mma_bf16(d_tmem, adesc + (uint64_t)(k * 2), bdesc0 + (uint64_t)(k * 2), idesc0, accum);
            if (n1 > 0)
              mma_bf16(d_tmem + SK_BN, adesc + (uint64_t)(k * 2), bdesc1 + (uint64_t)(k * 2),
                       idesc1, accum);
          }
          mma_commit(smem_u32(&empty[stage]));  // stage reusable once these MMAs finish
          if (F8) {
            mma_commit(smem_u32(&cempty[cst]));  // and the bf16 buffer
            if (++cst == p.cstages) {
              cst = 0;
              cphase ^= 1u;
            }
          }
          if (++stage == XS) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) mma_commit(smem_u32(&tfull[acc]));  // accumulator ready for the epilogue
      }
      if (++acc == p.acc_bufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    });
    // every MMA this thread issued has completed before TMEM is released
    mma_commit(smem_u32(drain));
    if (!mbar_wait_bounded(smem_u32(drain), 0)) report_error(p.err, kErrTimeoutDrain);
  } else if (warp >= SK_EPI_WARP0 && warp < SK_EPI_WARP0 + 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                // TMEM lane quadrant this warp may access
    const int64_t t = q * 32 + lane;       // this thread's token
    const bool has_tokens = q * 32 < p.M;  // warp-uniform
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    SK_FOR_EACH_TILE(tl, {
      if (ok) {
        // all lanes wait, then agree: tcgen05.ld is warp-collective
        ok = mbar_wait_bounded(smem_u32(&tfull[acc]), acc_phase);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && lane == 0) report_error(p.err, kErrTimeoutEpilogue);
      }
      if (ok) {
        tc_fence_after();
        const uint32_t taddr =
            tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.acc_stride);
        // Only lanes t < M hold a token; the other lanes' accumulator rows
        // come from shared memory that is not this call's X (whatever the
        // ring held), so they only take part in the warp-collective TMEM
        // loads: no arithmetic and no stores.  Accumulator columns are read
        // 16 (gate and up: 2 x 16) at a time with one wait.
        const bool live = t < p.M;
        if (has_tokens && p.csplit) {
          // column K split: this rank's partials of the cluster's features
          // -> shared memory, at the feature's offset in the cluster's range
          // (SwiGLU: up partials tile_cap further)
          for (int i = 0; i < tl.n; ++i) {
            const Piece& pc = tl.pc[i];
            const int64_t fl0 = p.fo[pc.shard] + pc.loc - f0;
#pragma unroll 1
            for (int j0 = 0; j0 < pc.c; j0 += 16) {
              float v[16], u[16];
              const uint32_t tg = taddr + (uint32_t)(pc.slot + j0);
              if (swiglu)
                tmem_ld16x2(tg, taddr + (uint32_t)(tl.rows + pc.slot + j0), v, u);
              else
                tmem_ld16(tg, v);
              if (!live) continue;
              const int valid = pc.c - j0 < 16 ? pc.c - j0 : 16;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int64_t o = t * SK_RED_PITCH + fl0 + j0 + j;
                if (j < valid &&
                    TP_CHECK(p.err, (o + (swiglu ? p.tile_cap : 0) + 1) * 4 <= p.red_bytes)) {
                  red[o] = v[j];
                  if (swiglu) red[o + p.tile_cap] = u[j];
                }
              }
            }
          }
        } else if (has_tokens && p.row && p.cs > 1) {
          // this rank's partial sum -> shared memory, for the cluster reduction
          const int c = tl.pc[0].c;
#pragma unroll 1
          for (int j0 = 0; j0 < c; j0 += 16) {
            float v[16];
            tmem_ld16(taddr + (uint32_t)j0, v);
            if (live &&
                TP_CHECK(p.err, (int64_t)(t * SK_RED_PITCH + j0 + 16) * 4 <= p.ring_bytes)) {
              if (F8) {
                // this CTA's partial belongs to shard rshard: its row scales
                const float* sc = p.wscale[rshard] + tl.pc[0].loc + j0;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (j0 + j < c) v[j] *= __ldg(sc + j);
              }
              float4* dst = reinterpret_cast<float4*>(red + t * SK_RED_PITCH + j0);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
          }
        } else if (has_tokens) {
          for (int i = 0; i < tl.n; ++i) {
            const Piece& pc = tl.pc[i];
            const int64_t base = (p.row ? 0 : p.yoff[pc.shard]) + t * p.ldy;
            const float* bias = p.row ? p.bias[0] : (swiglu ? nullptr : p.bias[pc.shard]);
            // FP8 mode: scales of the piece's (gate) rows; up rows G further
            const float* sc = nullptr;
            if (F8)
              sc = p.wscale[p.row ? rshard : pc.shard] +
                   (swiglu ? (pc.loc / G) * 2 * G + pc.loc % G : pc.loc);
            // 16 columns per step (8 in FP8 mode, whose 704 threads leave
            // fewer registers each)
            constexpr int CH = F8 ? 8 : 16;
#pragma unroll 1
            for (int j0 = 0; j0 < pc.c; j0 += CH) {
              // columns [slot + j0, slot + j0 + CH) lie inside the piece's
              // slot (slots are multiples of 16 wide)
              float v[CH], u[CH];
              const uint32_t tg = taddr + (uint32_t)(pc.slot + j0);
              const uint32_t tu = taddr + (uint32_t)(tl.rows + pc.slot + j0);
              if constexpr (CH == 16) {
                if (swiglu)
                  tmem_ld16x2(tg, tu, v, u);
                else
                  tmem_ld16(tg, v);
              } else {
                tmem_ld8(tg, v);
                if (swiglu) tmem_ld8(tu, u);
              }
              if (!live) continue;
              const int valid = pc.c - j0 < CH ? pc.c - j0 : CH;
              if (F8) {
#pragma unroll
                for (int j = 0; j < CH; ++j)
                  if (j < valid) {
                    v[j] *= __ldg(sc + j0 + j);
                    if (swiglu) u[j] *= __ldg(sc + G + j0 + j);
                  }
              }
              if (swiglu) {
#pragma unroll
                for (int j = 0; j < CH; ++j) v[j] = act_silu(v[j]) * u[j];
              } else {
                if (bias) {
#pragma unroll
                  for (int j = 0; j < CH; ++j)
                    if (j < valid) v[j] += __ldg(bias + pc.loc + j0 + j);
                }
                if (!p.row && p.act == TP_ACT_GELU_ERF) {
#pragma unroll
                  for (int j = 0; j < CH; ++j) v[j] = act_gelu_erf(v[j]);
                }
              }
              if (!TP_CHECK(p.err, base + pc.loc + j0 + valid <= p.y_extent)) continue;
              if constexpr (CH == 16)
                store_row16(p.Y, p.ydt, base, pc.loc + j0, valid, v);
              else
                store_row8(p.Y, p.ydt, base, pc.loc + j0, valid, v);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
      }
      if (++acc == p.acc_bufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    });
  }

  if (F8 && warp >= SK_CONV_WARP0) {
    // ------------------------------------------------------------ converters
    // A raw stage holds SK_KPR k-blocks of each tile row (rows SK_RAW_ROW_BYTES
    // apart); each k-block becomes one bf16 B tile in the 128-byte swizzled
    // K-major layout the MMA's descriptor expects.  k-block n of the CTA's
    // sequence is converted by group n mod 2 into buffer n mod 2.  Thread gt
    // of a group owns 16-byte chunk c4 = gt mod 4 of a k-block (codes
    // [16 c4, 16 c4 + 16)) in rows gt / 4, gt / 4 + SK_GROUP_THREADS / 4, ...;
    // it writes them as bf16 chunks 2 c4 and 2 c4 + 1 of the row, each at
    // chunk position c ^ (row mod 8).  Every converter warp releases each raw
    // stage once, whether or not its group had a k-block in it.
    const int cw = warp - SK_CONV_WARP0;
    const int grp = cw / SK_GROUP_WARPS;
    const int gt = (cw % SK_GROUP_WARPS) * 32 + lane;
    const int row0 = gt >> 2, c4 = gt & 3, sw = row0 & 7;
    constexpr int RSTEP = SK_GROUP_THREADS / 4;
    const uint32_t src0 = (uint32_t)(row0 * SK_RAW_ROW_BYTES + c4 * 16);
    const uint32_t dlo0 = (uint32_t)(row0 * SK_ROW_BYTES + (((2 * c4) ^ sw) << 4));
    const uint32_t dhi0 = (uint32_t)(row0 * SK_ROW_BYTES + (((2 * c4 + 1) ^ sw) << 4));
    uint8_t* const mybuf = sW + (size_t)grp * p.w_stage_bytes;
    int rs = 0;
    uint32_t rphase = 0, cphase = 0;
    int64_t n = 0;  // k-blocks of the CTA's sequence before this raw stage
    bool ok = true;
    SK_FOR_EACH_TILE(tl, {
      if (ok) {
        const int nrows = swiglu ? 2 * tl.rows : tl.rows;
        if (!TP_CHECK(p.err, nrows * SK_RAW_ROW_BYTES <= p.raw_stage_bytes &&
                                 nrows * SK_ROW_BYTES <= p.w_stage_bytes))
          ok = false;
        for (int kb = tl.kb0; kb < tl.kb1 && ok; kb += SK_KPR) {
          const int nsub = tl.kb1 - kb < SK_KPR ? tl.kb1 - kb : SK_KPR;
          bool got = mbar_wait_bounded(smem_u32(&rfull[rs]), rphase);
          got = __all_sync(0xffffffffu, got);
          if (!got) {
            if (lane == 0) report_error(p.err, kErrTimeoutConvert);
            ok = false;
            break;
          }
          for (int j = 0; j < nsub; ++j) {
            if ((int)((n + j) % SK_CONV_GROUPS) != grp) continue;
            bool gc = mbar_wait_bounded(smem_u32(&cempty[grp]), cphase ^ 1u);
            gc = __all_sync(0xffffffffu, gc);
            if (!gc) {
              if (lane == 0) report_error(p.err, kErrTimeoutConvert);
              ok = false;
              break;
            }
            const uint8_t* src = sR + (size_t)rs * p.raw_stage_bytes + src0 + j * SK_BK;
            uint8_t* dst = mybuf;
#pragma unroll 4
            for (int r = row0; r < nrows; r += RSTEP) {
              const uint4 q = *reinterpret_cast<const uint4*>(src);
              uint4 lo, hi;
              e4m3x4_to_bf16x4(q.x, lo.x, lo.y);
              e4m3x4_to_bf16x4(q.y, lo.z, lo.w);
              e4m3x4_to_bf16x4(q.z, hi.x, hi.y);
              e4m3x4_to_bf16x4(q.w, hi.z, hi.w);
              *reinterpret_cast<uint4*>(dst + dlo0) = lo;
              *reinterpret_cast<uint4*>(dst + dhi0) = hi;
              src += RSTEP * SK_RAW_ROW_BYTES;
              dst += RSTEP * SK_ROW_BYTES;
            }
            fence_proxy_async_smem();  // the MMA reads these writes through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&cfull[grp]));
            cphase ^= 1u;
          }
          if (!ok) break;
          n += nsub;
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&rempty[rs]));  // codes read: the raw stage is free
          if (++rs == S) {
            rs = 0;
            rphase ^= 1u;
          }
        }
      }
    });
  }

  __syncthreads();
  if (p.row && p.cs > 1) {
    // ---------------------------------------------------------- cluster reduction
    // Every thread of every CTA of the cluster passes both barriers, whatever
    // happened above.
    cluster_sync_all();
    const Tile tl = row_tile(p, rank);
    const int c = tl.pc[0].c;
    const int64_t loc = tl.pc[0].loc;
    const int w = (p.tile_cap + p.cs - 1) / p.cs;  // outputs per rank
    const int j_lo = rank * w;
    const int j_hi = (int)imin((int64_t)j_lo + w, c);
    const float* bias = p.bias[0];
    const uint32_t red_s = smem_u32(red);
    if (j_hi > j_lo) {
      const int span = j_hi - j_lo;
      const int64_t items = p.M * span;
      for (int64_t it = threadIdx.x; it < items; it += blockDim.x) {
        const int64_t tok = it / span;
        const int j = j_lo + (int)(it - tok * span);
        const uint32_t off = (uint32_t)((tok * SK_RED_PITCH + j) * 4);
        float sum = 0.0f;
        for (int r = 0; r < p.cs; ++r) sum += dsmem_ld_f32(dsmem_addr(red_s + off, (uint32_t)r));
        if (bias) sum += __ldg(bias + loc + j);
        if (TP_CHECK(p.err, tok * p.ldy + loc + j < p.y_extent))
          store_out(p.Y, p.ydt, tok * p.ldy + loc + j, sum);
      }
    }
    cluster_sync_all();  // no CTA leaves while a peer still reads its buffer
  }
  if (p.csplit) {
    // ---------------------------------------------- column K split: reduction
    // CTA r of the cluster finishes features [r w, (r + 1) w) of its range:
    // the cs partials in rank order, then bias / activation, one rounding.
    // Every thread of every CTA passes both barriers.
    cluster_sync_all();
    const int64_t nf = f1 - f0;
    const int64_t w = (nf + p.cs - 1) / p.cs;
    const int64_t lo = (int64_t)rank * w;
    const int64_t hi = imin(lo + w, nf);
    const uint32_t red_s = smem_u32(red);
    if (hi > lo) {
      const int64_t span = hi - lo;
      const int64_t items = p.M * span;
      for (int64_t it = threadIdx.x; it < items; it += blockDim.x) {
        const int64_t tok = it / span;
        const int64_t fl = lo + (it - tok * span);
        const int64_t g = f0 + fl;
        int sh = 0;
        while (sh + 1 < p.tp && p.fo[sh + 1] <= g) ++sh;
        const int64_t loc = g - p.fo[sh];
        const uint32_t off = (uint32_t)((tok * SK_RED_PITCH + fl) * 4);
        float v = 0.0f;
        for (int r = 0; r < p.cs; ++r) v += dsmem_ld_f32(dsmem_addr(red_s + off, (uint32_t)r));
        if (swiglu) {
          const uint32_t offu = off + (uint32_t)(p.tile_cap * 4);
          float u = 0.0f;
          for (int r = 0; r < p.cs; ++r) u += dsmem_ld_f32(dsmem_addr(red_s + offu, (uint32_t)r));
          v = act_silu(v) * u;
        } else {
          if (p.bias[sh]) v += __ldg(p.bias[sh] + loc);
          if (p.act == TP_ACT_GELU_ERF) v = act_gelu_erf(v);
        }
        const int64_t yo = p.yoff[sh] + tok * p.ldy + loc;
        if (TP_CHECK(p.err, yo < p.y_extent)) store_out(p.Y, p.ydt, yo, v);
      }
    }
    cluster_sync_all();  // no CTA leaves while a peer still reads its buffer
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, SK_TMEM_COLS);
  }
}

#undef SK_FOR_EACH_TILE

template <bool F8>
tp_status prepare_skinny_mode(const LinearProblem& p, Launch* L) {
  if (p.xdt != TP_BF16 || p.M < 1 || p.M > kSkinnyMaxTokens) return TP_ERR_UNSUPPORTED;
  if (F8 && p.row && p.tp > SK_MAX_CLUSTER) return TP_ERR_UNSUPPORTED;
  SkinnyParams sp{};
  sp.err = device_error_word();
  if (!sp.err) return TP_ERR_CUDA;
  const int xrows = (int)((p.M + 7) / 8 * 8);
  const int64_t es = 2;
  if (p.row) {
    for (int i = 0; i < p.tp; ++i) {
      const void* xi = static_cast<const char*>(p.X) + (int64_t)i * p.x_shard_off * es;
      if (!make_tma_map_bf16(&sp.tmX[i], xi, (uint64_t)p.K, (uint64_t)p.M,
                             (uint64_t)(p.ldx * es), (uint32_t)xrows))
        return TP_ERR_CUDA;
    }
  } else if (!make_tma_map_bf16(&sp.tmX[0], p.X, (uint64_t)p.K, (uint64_t)p.M,
                                (uint64_t)(p.ldx * es), (uint32_t)xrows)) {
    return TP_ERR_CUDA;
  }
  for (int i = 0; i < p.tp; ++i) {
    const uint64_t rows = (uint64_t)(p.row ? p.w_rows : p.wr[i]);
    bool ok;
    if (F8) {  // e4m3 codes: one byte per weight
      ok = make_tma_map_u8(&sp.tmW16[i], p.W[i], (uint64_t)p.K, rows, (uint64_t)p.K,
                           SK_RAW_ROW_BYTES, 16, false) &&
           make_tma_map_u8(&sp.tmW64[i], p.W[i], (uint64_t)p.K, rows, (uint64_t)p.K,
                           SK_RAW_ROW_BYTES, 64, false);
    } else {
      ok = make_tma_map_bf16(&sp.tmW16[i], p.W[i], (uint64_t)p.K, rows, (uint64_t)(p.K * es), 16) &&
           make_tma_map_bf16(&sp.tmW64[i], p.W[i], (uint64_t)p.K, rows, (uint64_t)(p.K * es), 64);
    }
    if (!ok) return TP_ERR_CUDA;
  }
  for (int i = 0; i < TP_MAX_TP; ++i) {
    sp.bias[i] = p.bias[i];
    sp.wscale[i] = F8 ? p.wscale[i] : nullptr;
  }
  sp.Y = p.Y;
  sp.ldy = p.ldy;
  sp.y_extent = output_extent(p);
  for (int i = 0; i <= p.tp; ++i) sp.fo[i] = p.fo[i];
  for (int i = 0; i < p.tp; ++i) sp.yoff[i] = p.yoff[i];
  sp.M = p.M;
  sp.feat_total = p.row ? p.n_out : p.fo[p.tp];
  sp.tp = p.tp;
  sp.row = p.row ? 1 : 0;
  sp.act = p.act;
  sp.ydt = p.ydt;
  sp.xrows = xrows;
  sp.x_stage_bytes = xrows * SK_ROW_BYTES;
  sp.kb_per_shard = (int)((p.K + SK_BK - 1) / SK_BK);
  sp.kb_total = sp.kb_per_shard * (p.row ? p.tp : 1);

  const int sms = sm_count();
  int grid = 1;
  sp.cs = 1;
  sp.csplit = 0;
  int resident[SK_MAX_CLUSTER + 1];
  if (p.row) {
    // Output tiles of bn; clusters of cs CTAs split each tile's K loop so
    // that tiles x cs fills the SMs (each CTA keeps at least one k-block).
    // FP8 mode: each CTA's k-range lies inside one shard (its partial is
    // scaled by that shard's row scales): tp x j CTAs, j per shard.
    const int unit = F8 ? p.tp : 1;
    resident_clusters(reinterpret_cast<const void*>(skinny_kernel<F8>),
                      F8 ? SK_THREADS_F8 : SK_THREADS, SK_SMEM_MAX, SK_MAX_CLUSTER, unit, resident);
    const decode::RowTiling rt = decode::choose_row_tiling(
        p.n_out, sp.kb_total, F8 ? sp.kb_per_shard : sp.kb_total, sms, SK_MAX_CLUSTER, unit,
        resident);
    if (rt.tiles * rt.cs > INT32_MAX) return TP_ERR_BAD_SHAPE;
    sp.cs = rt.cs;
    sp.tile_cap = rt.bn;
    grid = (int)(rt.tiles * rt.cs);
  } else {
    const int64_t units = (sp.feat_total + SK_GRAIN - 1) / SK_GRAIN;
    grid = (int)std::max<int64_t>(1, std::min<int64_t>(units, sms));
  }
  // B tile: the row side's tile of outputs; on the column side as many
  // features (rows) as the widest CTA range, up to 256 (SwiGLU: gate + up
  // rows).
  const bool swiglu = !p.row && p.act == TP_ACT_SWIGLU;
  int tile_rows = p.row ? sp.tile_cap : SK_BN;
  if (!p.row) {
    const int64_t units = (sp.feat_total + SK_GRAIN - 1) / SK_GRAIN;
    const int64_t max_range = (units + grid - 1) / grid * SK_GRAIN;
    // FP8 mode: at most 256 rows (gate + up) per tile
    const int64_t cap = (F8 && swiglu) ? SK_BN / 2 : SK_BN;
    sp.tile_cap = (int)std::min<int64_t>(cap, max_range);
    tile_rows = swiglu ? 2 * sp.tile_cap : sp.tile_cap;
    if (!F8 && tile_rows < SK_SPLIT_ROWS && p.M <= SK_SPLIT_MAX_TOKENS) {
      // K split over clusters: tiles of 256 weight rows (SwiGLU: 128
      // features, gate and up)
      const int wf = swiglu ? SK_BN / 2 : SK_BN;
      resident_clusters(reinterpret_cast<const void*>(skinny_kernel<F8>), SK_THREADS,
                        SK_SMEM_MAX, SK_MAX_CLUSTER, 1, resident);
      const decode::RowTiling ct = decode::choose_row_tiling(
          sp.feat_total, sp.kb_total, sp.kb_total / SK_SPLIT_MIN_KB, sms, SK_MAX_CLUSTER, 1,
          resident, wf);
      if (ct.cs >= 2 && ct.tiles * ct.cs <= INT32_MAX) {
        sp.csplit = 1;
        sp.cs = ct.cs;
        sp.tile_cap = wf;
        tile_rows = swiglu ? 2 * wf : wf;
        grid = (int)(ct.tiles * ct.cs);
      }
    }
  }
  sp.w_stage_bytes = tile_rows * SK_ROW_BYTES;
  sp.raw_stage_bytes = F8 ? tile_rows * SK_RAW_ROW_BYTES : 0;
  sp.cstages = F8 ? SK_CSTAGES : 0;
  sp.acc_stride = (tile_rows + 31) / 32 * 32;
  sp.acc_bufs = (SK_ACC_BUFS * sp.acc_stride <= SK_TMEM_COLS) ? SK_ACC_BUFS : 1;
  // column K split: the partial sums of up to SK_SPLIT_MAX_TOKENS tokens,
  // after the barriers
  const int bar_bytes = (SK_BAR_BYTES + 15) / 16 * 16;
  sp.red_bytes = sp.csplit ? (int)p.M * SK_RED_PITCH * 4 : 0;
  const int avail = SK_SMEM_MAX - 1024 - bar_bytes - sp.red_bytes;
  // bf16: a stage is the X box and the weight rows.  FP8: a stage is the raw
  // codes; the X ring (about 32 KB) and the bf16 buffers are fixed.
  sp.xstages = F8 ? std::max(2, std::min(SK_MAX_STAGES, 32768 / sp.x_stage_bytes)) : 0;
  const int per_stage = F8 ? sp.raw_stage_bytes : sp.x_stage_bytes + sp.w_stage_bytes;
  const int fixed = F8 ? sp.xstages * sp.x_stage_bytes + sp.cstages * sp.w_stage_bytes : 0;
  const int stages = std::min(SK_MAX_STAGES, (avail - fixed) / per_stage);
  if (stages < 2) return TP_ERR_UNSUPPORTED;
  sp.stages = stages;
  const int ring = stages * per_stage + fixed;
  sp.ring_bytes = ring;
  const int x_ring_stages = F8 ? sp.xstages : stages;
  // The MMA reads a full 128-row A tile from each X stage: the read past the
  // last X stage runs into the stages after the X ring (weights, or codes in
  // FP8 mode), which must be there.  The row side's reduction buffer reuses
  // the ring.
  if ((x_ring_stages - 1) * sp.x_stage_bytes + SK_A_BYTES > ring) return TP_ERR_UNSUPPORTED;
  if (p.row && sp.cs > 1 && (int64_t)xrows * SK_RED_PITCH * 4 > ring) return TP_ERR_UNSUPPORTED;
  sp.red_off = sp.csplit ? ring + bar_bytes : 0;
  const int smem = 1024 + ring + bar_bytes + sp.red_bytes;

  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(skinny_kernel<F8>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, SK_SMEM_MAX);
  });
  if (attr_err != cudaSuccess) return TP_ERR_CUDA;
  L->kernel = reinterpret_cast<const void*>(skinny_kernel<F8>);
  L->grid = dim3((unsigned)grid);
  L->block = dim3(F8 ? SK_THREADS_F8 : SK_THREADS);
  L->smem = (size_t)smem;
  L->cluster = (unsigned)sp.cs;
  L->pdl = true;
  L->set_params(sp);
  return TP_OK;
}

}  // namespace

tp_status prepare_skinny(const LinearProblem& p, Launch* L) {
  return p.fp8 ? prepare_skinny_mode<true>(p, L) : prepare_skinny_mode<false>(p, L);
}

}  // namespace tpla
