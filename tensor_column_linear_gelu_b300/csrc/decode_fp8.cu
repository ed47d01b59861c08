// decode_fp8.cu -- tcgen05 decode kernel for FP8 (e4m3) weights with the
// widened weights in tensor memory.
//
// A decode-shaped call reads every weight byte once, so e4m3 weights (one
// byte each, "Model Parallelism" (statistical-learning-notes), opening
// section) halve the bytes it streams.  The tensor core has no bf16 x e4m3
// form, so the codes are widened to bf16 on chip (exactly: every e4m3 value
// is a bf16 value).  Widening them into a shared-memory B tile costs about
// seven bytes of shared-memory traffic per code byte (TMA write, converter
// read and write, the MMA's operand reads), and that traffic, not HBM, set
// the pace of the shared-memory design.  Here the converters write the
// widened weights into TENSOR MEMORY as the MMA's A operand instead
// (tcgen05.st), and the tokens are the small N side read from shared memory:
//   D[128 weight rows, np tokens] += A[128 rows, 16 k] . X[np tokens, 16 k]^T
// per tcgen05.mma (M=128, N=np = tokens rounded up to 16, K=16).  An M=128,
// K=16 MMA takes about 112 cycles on this part whatever N is (measured), so a
// CTA streams at most 128 x 16 codes per 112 cycles, about 0.85 of its share
// of HBM bandwidth; shared memory now carries only the codes (TMA write,
// converter read) and the small X boxes.
//
//   column-parallel:  as the bf16 decode kernel (skinny.cu): CTA b owns an
//                     equal range of output features, cut into pieces at
//                     shard and gate/up-group boundaries and packed at 16-row
//                     slots into tiles of up to 512 rows (SwiGLU: up to 256
//                     features, gate slots then up slots).  A tile's rows are
//                     four MMA groups of 128 TMEM lanes: plain slot s is
//                     group s / 128, lane s mod 128; SwiGLU gate slot s is
//                     group s / 128 and its up slot group 2 + s / 128, the
//                     SAME lane, so one epilogue thread holds both.  Every
//                     output accumulates over all of K in one TMEM column:
//                     bit-identical to tp = 1.
//   row-parallel:     tiles of 256 outputs (groups 0 and 1), clusters of
//                     tp x j CTAs each streaming a k-range inside one shard;
//                     each partial is scaled by its shard's row scales, then
//                     the cluster adds the partials in rank order through
//                     distributed shared memory, plus the bias once.
//
// Roles (736 threads, one CTA per SM):
//   warp 0      TMA producer: code boxes (128 codes = two k-blocks per row,
//               128-byte swizzle, one box per lane) into a ring of raw stages,
//               and one X box {64, np} per k-block into the X ring;
//   warp 1      TMEM allocation (512 columns: A buffers in columns 0-255 --
//               two of 4 groups x 32 columns for column tiles, four of 2
//               groups for row tiles -- then D at column 256, np columns per
//               group) and the first MMA thread; warp 22 holds the second;
//   warps 2-5   epilogue (lane quarter = warp mod 4): scale, bias,
//               activation, stores; row side: partials to shared memory;
//   warps 6-21  converters: warp w widens group (w - 6) / 4, lane quarter
//               w mod 4 -- each thread one weight row, 64 codes per k-block:
//               four swizzled 16-byte shared loads, 32 bf16x2 words, one
//               tcgen05.st of 32 columns into A buffer n mod (A buffers).
// Every wait is bounded (sync.cuh); a wait that gives up records the error
// and that role stops issuing work, and every thread still reaches the
// cluster barriers and the TMEM release.
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

constexpr int TF_EPI_WARP0 = 2;
constexpr int TF_CONV_WARP0 = 6;
constexpr int TF_CONV_WARPS = 16;
constexpr int TF_ISSUERS = 2;              // MMA threads: warp 1, then warps TF_MMA2_WARP ..
constexpr int TF_MMA2_WARP = TF_CONV_WARP0 + TF_CONV_WARPS;
constexpr int TF_THREADS = 32 * (TF_MMA2_WARP + TF_ISSUERS - 1);
constexpr int TF_GROUPS = 4;               // 128-lane MMA groups per tile (512 rows)
constexpr int TF_BK = 64;                  // k per k-block (four K=16 MMAs)
constexpr int TF_KPR = 2;                  // k-blocks per raw stage
constexpr int TF_RAW_ROW = TF_BK * TF_KPR;  // 128 bytes of codes per raw row
constexpr int TF_X_ROW = 128;              // bytes per staged X row (64 bf16)
constexpr int TF_A_COLS = 32;              // TMEM columns of one group's A k-block
// A buffers: 256 TMEM columns hold 256 / (32 x groups per tile) k-blocks of
// A -- two for 4-group column tiles, four for the row side's 2-group tiles --
// so the converters can run that many k-blocks ahead of the MMAs.
constexpr int TF_A_REGION = 256;
constexpr int TF_MAX_ABUFS = 4;
constexpr int TF_D_BASE = TF_A_REGION;
constexpr int TF_MAX_NP = 64;
constexpr int TF_TMEM_COLS = 512;
static_assert(TF_D_BASE + TF_GROUPS * TF_MAX_NP <= TF_TMEM_COLS, "TMEM budget");
static_assert(TF_A_REGION / (TF_A_COLS * 2) <= TF_MAX_ABUFS, "A buffers of 2-group tiles");
static_assert(TF_CONV_WARPS == 4 * TF_GROUPS, "one converter warp per (group, lane quarter)");
constexpr int TF_MAX_STAGES = 16;
constexpr int TF_MAX_CLUSTER = kSkinnyMaxCluster;
constexpr int TF_RED_PITCH = SK_BN + 4;    // floats per token row of a reduction buffer
constexpr int TF_NUM_BARS = 4 * TF_MAX_STAGES + 2 * TF_MAX_ABUFS + 3;
constexpr int TF_BAR_BYTES = TF_NUM_BARS * 8 + 16;
constexpr int TF_SMEM_MAX = 232448;

struct Fp8TmemParams {
  CUtensorMap tmX[TP_MAX_TP];    // column: [0] = X; row: X_i.  bf16, box {64, np}, SW128
  CUtensorMap tmQ16[TP_MAX_TP];  // codes of W_i, box {128, 16}, SW128
  CUtensorMap tmQ64[TP_MAX_TP];  // codes of W_i, box {128, 64}, SW128
  const float* bias[TP_MAX_TP];
  const float* wscale[TP_MAX_TP];  // scale of each row of W_i
  void* Y;
  int64_t y_extent;  // elements of Y this call may write (checked builds)
  unsigned int* err;
  int64_t ldy;
  int64_t fo[TP_MAX_TP + 1];     // column: shard i owns features [fo[i], fo[i+1])
  int64_t yoff[TP_MAX_TP];       // column: element offset of shard i's outputs in Y
  int64_t M, feat_total;         // feat_total: column fo[tp]; row n_out
  int tp, row, act, ydt;
  int np;                        // tokens rounded up to 16: the MMA's N, X box rows
  int x_stage_bytes, xstages;
  int raw_stage_bytes, stages;
  int tile_cap;                  // column: features (SwiGLU) or rows per tile
  int kb_per_shard, kb_total;
  int cs;                        // row side: CTAs per cluster splitting K
  int tgroups;                   // MMA groups a tile can use: 4 (column), 2 (row)
  int abufs;                     // A buffers: TF_A_REGION / (32 x tgroups)
  int ring_bytes;                // shared memory below the barriers (checked builds)
};

__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane, then wait for the
// stores to complete.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// MMA groups a tile uses: plain, groups [0, ng); SwiGLU, gate groups [0, ng)
// and up groups [2, 2 + ng), ng = the tile's slot rows / 128 rounded up.
__device__ __forceinline__ bool group_active(int g, int rows, bool swiglu) {
  const int ng = (rows + 127) / 128;
  return swiglu ? (g & 1) < ng : g < ng;
}

__global__ void __launch_bounds__(TF_THREADS, 1)
    fp8_tmem_kernel(const __grid_constant__ Fp8TmemParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int XS = p.xstages, S = p.stages;
  uint8_t* sX = smem;                                      // XS X stages
  uint8_t* sR = smem + (size_t)XS * p.x_stage_bytes;       // S raw code stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(sR + (size_t)S * p.raw_stage_bytes);
  uint64_t* full = bars;                            // X landed
  uint64_t* empty = bars + TF_MAX_STAGES;           // X consumed by the MMAs
  uint64_t* rfull = bars + 2 * TF_MAX_STAGES;       // codes landed
  uint64_t* rempty = bars + 3 * TF_MAX_STAGES;      // codes read by the converters
  uint64_t* cfull = bars + 4 * TF_MAX_STAGES;       // A buffer written (TMEM)
  uint64_t* cempty = cfull + TF_MAX_ABUFS;          // A buffer consumed by the MMAs
  uint64_t* tfull = cempty + TF_MAX_ABUFS;          // accumulators final
  uint64_t* tempty = tfull + 1;                     // accumulators read out
  uint64_t* drain = tempty + 1;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + TF_NUM_BARS);
  // Row side: after the K loop the ring is reused as red[token][TF_RED_PITCH].
  float* red = reinterpret_cast<float*>(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool swiglu = (!p.row && p.act == TP_ACT_SWIGLU);
  const int rank = p.row ? (int)cluster_ctarank() : 0;
  const int rshard = p.row ? (int)((int64_t)rank * p.tp / p.cs) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < XS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), TF_ISSUERS);  // one commit per MMA thread
    }
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&rfull[s]), 1);
      mbar_init(smem_u32(&rempty[s]), TF_CONV_WARPS);
    }
    for (int b = 0; b < p.abufs; ++b) {
      mbar_init(smem_u32(&cfull[b]), TF_CONV_WARPS);
      mbar_init(smem_u32(&cempty[b]), TF_ISSUERS);
    }
    mbar_init(smem_u32(tfull), TF_ISSUERS);
    mbar_init(smem_u32(tempty), 4);  // one arrive per epilogue warp
    mbar_init(smem_u32(drain), TF_ISSUERS);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    const int nx = p.row ? p.tp : 1;
    for (int i = 0; i < nx; ++i) prefetch_tmap(&p.tmX[i]);
    for (int i = 0; i < p.tp; ++i) {
      prefetch_tmap(&p.tmQ16[i]);
      prefetch_tmap(&p.tmQ64[i]);
    }
  }
  if (warp == 1) tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), TF_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int64_t f0 = 0, f1 = 0;
  if (!p.row) column_range(p, f0, f1);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Per raw stage (two k-blocks): lane 0 waits for the stage and arms its
    // barrier, lane 1 + b loads code box b of the tile; then lane 0 loads the
    // X boxes of those k-blocks, one per X stage.
    int xs = 0, rs = 0;
    uint32_t xphase = 0, rphase = 0;
    bool ok = true;
    const uint64_t pol_x = l2_policy_evict_last();
    const uint64_t pol_w = l2_policy_evict_first();
    SK_FOR_EACH_TILE(tl, {
      if (ok) {
        int piece = 0, half = 0, r = 0, h = 0;
        const bool has_box = lane > 0 && tile_box(tl, swiglu, lane - 1, piece, half, r, h);
        int64_t wrow = 0;   // first weight row of this lane's box in its shard buffer
        uint32_t woff = 0;  // its offset in the raw stage
        int wshard = 0;
        if (has_box) {
          const Piece& pc = tl.pc[piece];
          wrow = (swiglu ? (pc.loc / G) * 2 * G + pc.loc % G + half * G : pc.loc) + r;
          woff = (uint32_t)(pc.slot + half * tl.rows + r) * TF_RAW_ROW;
          wshard = pc.shard;
        }
        const bool mine =
            has_box && TP_CHECK(p.err, woff + (uint32_t)h * TF_RAW_ROW <= (uint32_t)p.raw_stage_bytes);
        uint32_t wbytes = 0;
        if (lane == 0) {
          for (int b = 0; b < tl.boxes; ++b) {
            int pi, hf, rr, hh;
            if (tile_box(tl, swiglu, b, pi, hf, rr, hh)) wbytes += (uint32_t)hh * TF_RAW_ROW;
          }
        }
        for (int kb = tl.kb0; kb < tl.kb1 && ok; kb += TF_KPR) {
          const int nsub = tl.kb1 - kb < TF_KPR ? tl.kb1 - kb : TF_KPR;
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
            const CUtensorMap* map = (h == 64) ? &p.tmQ64[sh] : &p.tmQ16[sh];
            // a box reaching past the range (or past K) reads codes nobody uses
            tma_load_2d_hint(smem_u32(sR + (size_t)rs * p.raw_stage_bytes) + woff, map,
                             kk * TF_BK, (int)wrow, wb, pol_w);
          }
          __syncwarp();
          if (++rs == S) {
            rs = 0;
            rphase ^= 1u;
          }
          for (int j = 0; j < nsub; ++j) {
            bool gx = true;
            if (lane == 0) gx = mbar_wait_bounded(smem_u32(&empty[xs]), xphase ^ 1u);
            gx = __shfl_sync(0xffffffffu, gx, 0);
            if (!gx) {
              if (lane == 0) report_error(p.err, kErrTimeoutProducer);
              ok = false;
              break;
            }
            if (lane == 0) {
              const uint32_t fb = smem_u32(&full[xs]);
              mbar_arrive_expect_tx(fb, (uint32_t)p.x_stage_bytes);
              tma_load_2d_hint(smem_u32(sX + (size_t)xs * p.x_stage_bytes), &p.tmX[rsh],
                               (kk + j) * TF_BK, 0, fb, pol_x);
            }
            __syncwarp();
            if (++xs == XS) {
              xs = 0;
              xphase ^= 1u;
            }
          }
        }
      }
    });
  } else if ((warp == 1 || warp >= TF_MMA2_WARP) && lane == 0) {
    // ------------------------------------------------------------ MMA issuers
    // TF_ISSUERS threads take turns over the active groups of every k-block, each waiting
    // on the same barriers and committing its own MMAs (the barriers count
    // both).  While one waits on a barrier or commits, the other's MMAs keep
    // the tensor core busy: the queue in front of it is short, and each
    // wait costs about as long as an MMA.
    const int issuer = warp == 1 ? 0 : 1 + warp - TF_MMA2_WARP;
    int xs = 0, buf = 0;
    uint32_t xphase = 0, cphase = 0, tphase = 0;
    bool ok = true;
    const uint32_t idesc = idesc_bf16_f32(128, p.np);
    SK_FOR_EACH_TILE(tl, {
      if (ok && !mbar_wait_bounded(smem_u32(tempty), tphase ^ 1u)) {
        report_error(p.err, kErrTimeoutMma);
        ok = false;
      }
      if (ok) {
        tc_fence_after();
        for (int kb = tl.kb0; kb < tl.kb1; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[xs]), xphase) ||
              !mbar_wait_bounded(smem_u32(&cfull[buf]), cphase)) {
            report_error(p.err, kErrTimeoutMma);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bdesc = sdesc_sw128(smem_u32(sX + (size_t)xs * p.x_stage_bytes));
          int nth = 0;  // index of the group among the tile's active groups
          for (int g = 0; g < TF_GROUPS; ++g) {
            if (!group_active(g, tl.rows, swiglu)) continue;
            if ((nth++ % TF_ISSUERS) != issuer) continue;
            if (!TP_CHECK(p.err, (buf * p.tgroups + g + 1) * TF_A_COLS <= TF_A_REGION &&
                                     TF_D_BASE + (g + 1) * p.np <= TF_TMEM_COLS))
              continue;
            const uint32_t a0 = tmem_base + (uint32_t)((buf * p.tgroups + g) * TF_A_COLS);
            const uint32_t d = tmem_base + (uint32_t)(TF_D_BASE + g * p.np);
#pragma unroll
            for (int k = 0; k < TF_BK / 16; ++k) {
              // A: 8 columns (16 bf16) per K=16 step; B: +32 bytes in the swizzle span
              const uint32_t accum = (kb > tl.kb0 || k > 0) ? 1u : 0u;
              mma_bf16_tmem_a(d, a0 + (uint32_t)(k * 8), bdesc + (uint64_t)(k * 2), idesc, accum);
            }
          }
          mma_commit(smem_u32(&empty[xs]));
          mma_commit(smem_u32(&cempty[buf]));
          if (++xs == XS) {
            xs = 0;
            xphase ^= 1u;
          }
          if (++buf == p.abufs) {
            buf = 0;
            cphase ^= 1u;
          }
        }
        if (ok) mma_commit(smem_u32(tfull));
      }
      tphase ^= 1u;
    });
    mma_commit(smem_u32(drain));
    if (!mbar_wait_bounded(smem_u32(drain), 0)) report_error(p.err, kErrTimeoutDrain);
  } else if (warp >= TF_EPI_WARP0 && warp < TF_EPI_WARP0 + 4) {
    // ------------------------------------------------------------ epilogue
    // Thread (quarter q, lane l) of group g holds slot g * 128 + 32 q + l
    // (SwiGLU: gate group g, up group g + 2, the same lane) for all tokens.
    const int q = warp & 3;
    uint32_t tphase = 0;
    bool ok = true;
    SK_FOR_EACH_TILE(tl, {
      if (ok) {
        ok = mbar_wait_bounded(smem_u32(tfull), tphase);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && lane == 0) report_error(p.err, kErrTimeoutEpilogue);
      }
      if (ok) {
        tc_fence_after();
        const int ng = (tl.rows + 127) / 128;  // groups holding outputs (SwiGLU: gate groups)
        for (int g = 0; g < ng; ++g) {
          const int s = g * 128 + q * 32 + lane;  // this thread's slot
          const bool valid = s < tl.rows;
          // the piece of the slot: shard, shard-local feature, and weight row
          int pi = 0;
          while (pi + 1 < tl.n && tl.pc[pi + 1].slot <= s) ++pi;
          const Piece& pc = tl.pc[pi];
          const bool in_piece = valid && s - pc.slot < pc.c;
          const int64_t n = pc.loc + (s - pc.slot);  // shard-local feature (row: output)
          float sc = 0.0f, scu = 0.0f, b = 0.0f;
          if (in_piece) {
            if (p.row) {
              sc = __ldg(p.wscale[rshard] + n);
            } else if (swiglu) {
              const int64_t wr = (n / G) * 2 * G + n % G;
              sc = __ldg(p.wscale[pc.shard] + wr);
              scu = __ldg(p.wscale[pc.shard] + wr + G);
            } else {
              sc = __ldg(p.wscale[pc.shard] + n);
              if (p.bias[pc.shard]) b = __ldg(p.bias[pc.shard] + n);
            }
            if (p.row && p.cs == 1 && p.bias[0]) b = __ldg(p.bias[0] + n);
          }
          const uint32_t lane_off = (uint32_t)(q * 32) << 16;
          const uint32_t dg = tmem_base + lane_off + (uint32_t)(TF_D_BASE + g * p.np);
          const uint32_t du = tmem_base + lane_off + (uint32_t)(TF_D_BASE + (g + 2) * p.np);
          for (int t0 = 0; t0 < p.np; t0 += 16) {
            float v[16];
            tmem_ld16(dg + (uint32_t)t0, v);
            if (swiglu) {
              float u[16];
              tmem_ld16(du + (uint32_t)t0, u);
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = act_silu(sc * v[j]) * (scu * u[j]);
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                v[j] = sc * v[j];
                if (!p.row || p.cs == 1) {
                  v[j] += b;
                  if (!p.row && p.act == TP_ACT_GELU_ERF) v[j] = act_gelu_erf(v[j]);
                }
              }
            }
            if (in_piece) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int64_t t = t0 + j;
                if (t >= p.M) break;
                if (p.row && p.cs > 1) {
                  if (TP_CHECK(p.err, (t * TF_RED_PITCH + s + 1) * 4 <= p.ring_bytes))
                    red[t * TF_RED_PITCH + s] = v[j];  // this rank's partial, slot = output
                } else {
                  const int64_t e = (p.row ? 0 : p.yoff[pc.shard]) + t * p.ldy + n;
                  if (TP_CHECK(p.err, e < p.y_extent)) store_out(p.Y, p.ydt, e, v[j]);
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(tempty));
      }
      tphase ^= 1u;
    });
  } else if (warp >= TF_CONV_WARP0 && warp < TF_CONV_WARP0 + TF_CONV_WARPS) {
    // ------------------------------------------------------------ converters
    const int cw = warp - TF_CONV_WARP0;
    const int g = cw >> 2;        // MMA group
    const int q = warp & 3;       // TMEM lane quarter this warp may access
    int rs = 0, buf = 0;
    uint32_t rphase = 0, cphase = 0;
    bool ok = true;
    SK_FOR_EACH_TILE(tl, {
      if (ok) {
        const bool active = group_active(g, tl.rows, swiglu);          // warp-uniform
        const int s = (swiglu ? (g & 1) : g) * 128 + q * 32 + lane;    // slot
        const int rraw = (swiglu && g >= 2) ? tl.rows + s : s;         // raw stage row
        const bool valid =
            active && s < tl.rows &&
            TP_CHECK(p.err, (int64_t)(rraw + 1) * TF_RAW_ROW <= p.raw_stage_bytes);
        const uint32_t tcol = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(g * TF_A_COLS);
        for (int kb = tl.kb0; kb < tl.kb1 && ok; kb += TF_KPR) {
          const int nsub = tl.kb1 - kb < TF_KPR ? tl.kb1 - kb : TF_KPR;
          bool got = mbar_wait_bounded(smem_u32(&rfull[rs]), rphase);
          got = __all_sync(0xffffffffu, got);
          if (!got) {
            if (lane == 0) report_error(p.err, kErrTimeoutConvert);
            ok = false;
            break;
          }
          const uint8_t* row = sR + (size_t)rs * p.raw_stage_bytes + (size_t)rraw * TF_RAW_ROW;
          for (int j = 0; j < nsub; ++j) {
            bool gc = mbar_wait_bounded(smem_u32(&cempty[buf]), cphase ^ 1u);
            gc = __all_sync(0xffffffffu, gc);
            if (!gc) {
              if (lane == 0) report_error(p.err, kErrTimeoutConvert);
              ok = false;
              break;
            }
            if (active && TP_CHECK(p.err, (buf * p.tgroups + g + 1) * TF_A_COLS <= TF_A_REGION)) {
              // k-block j of the row: 16-byte chunks 4j .. 4j+3, each stored at
              // chunk (c ^ (row mod 8)) by the 128-byte swizzle
              uint32_t w[32];
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                uint4 qv = make_uint4(0u, 0u, 0u, 0u);
                if (valid)
                  qv = *reinterpret_cast<const uint4*>(row + (((4 * j + c) ^ (rraw & 7)) << 4));
                e4m3x4_to_bf16x4(qv.x, w[8 * c + 0], w[8 * c + 1]);
                e4m3x4_to_bf16x4(qv.y, w[8 * c + 2], w[8 * c + 3]);
                e4m3x4_to_bf16x4(qv.z, w[8 * c + 4], w[8 * c + 5]);
                e4m3x4_to_bf16x4(qv.w, w[8 * c + 6], w[8 * c + 7]);
              }
              // word i = bf16 pair (k = 2i, 2i + 1), the lower k in the low half
              tmem_st32(tcol + (uint32_t)(buf * p.tgroups * TF_A_COLS), w);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&cfull[buf]));
            if (++buf == p.abufs) {
              buf = 0;
              cphase ^= 1u;
            }
          }
          if (!ok) break;
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&rempty[rs]));  // codes read: the stage is free
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
        const uint32_t off = (uint32_t)((tok * TF_RED_PITCH + j) * 4);
        float sum = 0.0f;
        for (int r = 0; r < p.cs; ++r) sum += dsmem_ld_f32(dsmem_addr(red_s + off, (uint32_t)r));
        if (bias) sum += __ldg(bias + loc + j);
        if (TP_CHECK(p.err, tok * p.ldy + loc + j < p.y_extent))
          store_out(p.Y, p.ydt, tok * p.ldy + loc + j, sum);
      }
    }
    cluster_sync_all();  // no CTA leaves while a peer still reads its buffer
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TF_TMEM_COLS);
  }
}

#undef SK_FOR_EACH_TILE

}  // namespace

tp_status prepare_decode_fp8(const LinearProblem& p, Launch* L) {
  if (!p.fp8 || p.xdt != TP_BF16 || p.M < 1 || p.M > kFp8TmemMaxTokens) return TP_ERR_UNSUPPORTED;
  if (p.row && p.tp > TF_MAX_CLUSTER) return TP_ERR_UNSUPPORTED;
  Fp8TmemParams fp{};
  fp.err = device_error_word();
  if (!fp.err) return TP_ERR_CUDA;
  const int np = (int)((p.M + 15) / 16 * 16);
  const int64_t es = 2;
  if (p.row) {
    for (int i = 0; i < p.tp; ++i) {
      const void* xi = static_cast<const char*>(p.X) + (int64_t)i * p.x_shard_off * es;
      if (!make_tma_map_bf16(&fp.tmX[i], xi, (uint64_t)p.K, (uint64_t)p.M,
                             (uint64_t)(p.ldx * es), (uint32_t)np))
        return TP_ERR_CUDA;
    }
  } else if (!make_tma_map_bf16(&fp.tmX[0], p.X, (uint64_t)p.K, (uint64_t)p.M,
                                (uint64_t)(p.ldx * es), (uint32_t)np)) {
    return TP_ERR_CUDA;
  }
  for (int i = 0; i < p.tp; ++i) {
    const uint64_t rows = (uint64_t)(p.row ? p.w_rows : p.wr[i]);
    if (!make_tma_map_u8(&fp.tmQ16[i], p.W[i], (uint64_t)p.K, rows, (uint64_t)p.K, TF_RAW_ROW,
                         16, true) ||
        !make_tma_map_u8(&fp.tmQ64[i], p.W[i], (uint64_t)p.K, rows, (uint64_t)p.K, TF_RAW_ROW,
                         64, true))
      return TP_ERR_CUDA;
  }
  for (int i = 0; i < TP_MAX_TP; ++i) {
    fp.bias[i] = p.bias[i];
    fp.wscale[i] = p.wscale[i];
  }
  fp.Y = p.Y;
  fp.ldy = p.ldy;
  fp.y_extent = output_extent(p);
  for (int i = 0; i <= p.tp; ++i) fp.fo[i] = p.fo[i];
  for (int i = 0; i < p.tp; ++i) fp.yoff[i] = p.yoff[i];
  fp.M = p.M;
  fp.feat_total = p.row ? p.n_out : p.fo[p.tp];
  fp.tp = p.tp;
  fp.row = p.row ? 1 : 0;
  fp.act = p.act;
  fp.ydt = p.ydt;
  fp.np = np;
  fp.kb_per_shard = (int)((p.K + TF_BK - 1) / TF_BK);
  fp.kb_total = fp.kb_per_shard * (p.row ? p.tp : 1);

  const int sms = sm_count();
  int grid = 1;
  fp.cs = 1;
  const bool swiglu = !p.row && p.act == TP_ACT_SWIGLU;
  int tile_rows = SK_BN;
  if (p.row) {
    // tiles of bn outputs; tp x j CTAs per cluster, each inside one shard
    int resident[TF_MAX_CLUSTER + 1];
    resident_clusters(reinterpret_cast<const void*>(fp8_tmem_kernel), TF_THREADS, TF_SMEM_MAX,
                      TF_MAX_CLUSTER, p.tp, resident);
    const RowTiling rt = choose_row_tiling(p.n_out, fp.kb_total, fp.kb_per_shard, sms,
                                           TF_MAX_CLUSTER, p.tp, resident);
    if (rt.tiles * rt.cs > INT32_MAX) return TP_ERR_BAD_SHAPE;
    fp.cs = rt.cs;
    grid = (int)(rt.tiles * rt.cs);
    fp.tile_cap = rt.bn;
    tile_rows = rt.bn;
  } else {
    const int64_t units = (fp.feat_total + SK_GRAIN - 1) / SK_GRAIN;
    grid = (int)std::max<int64_t>(1, std::min<int64_t>(units, sms));
    const int64_t max_range = (units + grid - 1) / grid * SK_GRAIN;
    // SwiGLU: up to 256 features (gate groups 0-1, up groups 2-3); plain: 512 rows
    const int64_t cap = swiglu ? 2 * 128 : TF_GROUPS * 128;
    fp.tile_cap = (int)std::min<int64_t>(cap, max_range);
    tile_rows = swiglu ? 2 * fp.tile_cap : fp.tile_cap;
  }
  fp.tgroups = p.row ? 2 : TF_GROUPS;
  fp.abufs = TF_A_REGION / (TF_A_COLS * fp.tgroups);
  fp.raw_stage_bytes = tile_rows * TF_RAW_ROW;
  fp.x_stage_bytes = np * TF_X_ROW;
  fp.xstages = std::max(2, std::min(TF_MAX_STAGES, 32768 / fp.x_stage_bytes));
  const int avail = TF_SMEM_MAX - 1024 - TF_BAR_BYTES;
  const int xring = fp.xstages * fp.x_stage_bytes;
  const int stages = std::min(TF_MAX_STAGES, (avail - xring) / fp.raw_stage_bytes);
  if (stages < 2) return TP_ERR_UNSUPPORTED;
  fp.stages = stages;
  const int ring = xring + stages * fp.raw_stage_bytes;
  fp.ring_bytes = ring;
  if (p.row && fp.cs > 1 && (int64_t)p.M * TF_RED_PITCH * 4 > ring) return TP_ERR_UNSUPPORTED;
  const int smem = 1024 + ring + TF_BAR_BYTES;

  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(fp8_tmem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    TF_SMEM_MAX);
  });
  if (attr_err != cudaSuccess) return TP_ERR_CUDA;
  L->kernel = reinterpret_cast<const void*>(fp8_tmem_kernel);
  L->grid = dim3((unsigned)grid);
  L->block = dim3(TF_THREADS);
  L->smem = (size_t)smem;
  L->cluster = (unsigned)fp.cs;
  L->set_params(fp);
  return TP_OK;
}

}  // namespace tpla
