// decode_f8mma.cu -- tcgen05 kernel for decode-shaped calls with e4m3 (FP8)
// weights: up to kF8MmaMaxTokens tokens against a large weight whose codes
// stream from HBM at one byte per weight.
//
// A call with a handful of tokens reads every weight byte once, so it is
// bound by the bytes it streams ("What is tensor parallelism?", "Why it helps
// when serving"); FP8 weights halve them ("Model Parallelism", opening
// section: about one byte per parameter).  What limits a tensor-core decode
// kernel besides the bytes is the MMA instruction rate: an M=128 tcgen05.mma
// takes roughly 110-130 cycles however small N is, so each instruction must
// cover many weights.  Here the codes are the MMA's N operand, straight from
// the TMA (no widening on chip): kind::f8f6f4, M=128, N<=256, K=32, so one
// instruction covers 256 x 32 weights.
//
// The tokens are the A operand, and kind::f8f6f4 needs them in an 8-bit
// format too.  They are split, exactly, into three e4m3 planes per token:
// with a per-token power-of-two scale 2^e (e chosen so that the token's
// largest |x| becomes u in [128, 256)), u = x * 2^-e,
//     hi  = e4m3(u),  lo = e4m3((u - hi) * 16),  lo2 = e4m3(((u - hi) * 16 - lo) * 16)
// (each e4m3() rounds to nearest even).  A bf16 value has 8 significant bits,
// hi keeps 4 and every residual fits the next plane, so u = hi + lo/16 +
// lo2/256 exactly for every |u| >= 2^-14 (|x| down to 2^-21 of the token's
// largest; smaller elements keep an absolute error below 2^-18 of it).  Token
// t uses A rows 4t .. 4t+2 (row 4t+3 is zero), so up to 32 tokens fill the
// 128 rows, and the three planes accumulate into TMEM lanes 4t .. 4t+2 of the
// same columns.  The epilogue combines them, y = s_n * 2^e * (a_hi + a_lo/16
// + a_lo2/256) with s_n the weight row's scale: the dot product is that of
// the exact bf16 tokens with the exact e4m3 weights, accumulated by the
// tensor core in fp32.
//
//   column-parallel:  Y_i = act(s * (X . Q_i^T) + b_i); CTA b of a persistent
//                     grid owns output features [b*F/grid, (b+1)*F/grid) in
//                     16-feature units, packed as pieces at 16-row slots of a
//                     B tile of up to 512 code rows (two MMAs of N <= 256 per
//                     k-step; SwiGLU: gate rows, then the up rows at the same
//                     slots).  Every output accumulates over all of K in one
//                     TMEM column and every CTA's token scales come from all
//                     of K, so sharded results are bit-identical to tp = 1.
//   row-parallel:     Y = sum_i s_i * (X_i . Q_i^T) + b; output tiles of 256,
//                     each split over a cluster of tp x j CTAs whose k-ranges
//                     lie inside one shard.  A CTA's partial is scaled by its
//                     shard's row scales (and its token scales, taken over its
//                     own k-range) before the cluster adds the partials in
//                     rank order through distributed shared memory, then the
//                     bias once.
// ("Understanding Tensor Parallelism for Multi-GPU LLM Serving", "How Tensor
// Parallelism Works Under the Hood"; "Tensor parallel serving",
// "Column-parallel and row-parallel layers, paired".)
//
// Roles (320 threads, one CTA per SM):
//   warp 0      TMA producer: the tile's code rows, 128 codes (one k-block)
//               wide, as 64-row and 16-row boxes with the 128-byte swizzle,
//               one box per lane.
//   warp 1      TMEM allocation (512 columns) and the single MMA-issuing thread.
//   warps 2-5   epilogue: TMEM lane quadrant q holds tokens 8q .. 8q+7; the
//               four lanes of a token combine its planes with two butterfly
//               shuffles and then each finishes a quarter of the columns.
//   warps 6-9   converters: first the token scales (max |x| over the CTA's
//               k-range), then per k-block the three planes of every token,
//               written in the 128-byte swizzled K-major layout the MMA's
//               descriptor expects.
// Two rings advance together, one stage per k-block: code stages (filled by
// the TMA) and plane stages (filled by the converters); the MMAs' commit
// releases both.
//
// Every mbarrier wait is bounded (sync.cuh); a wait that gives up records the
// failure in the device error word and that role stops.  Every thread of every
// CTA still reaches both cluster barriers.
#include <cuda.h>
#include <cuda_fp8.h>

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

constexpr int FM_THREADS = 320;
constexpr int FM_EPI_WARP0 = 2;
constexpr int FM_CONV_WARP0 = 6;
constexpr int FM_CONV_THREADS = 128;
// Conversion tasks (8 k of one token) per converter thread and k-block are a
// template parameter, CT = ceil(16 x token slots / 128): 1 up to 8 tokens,
// 2 up to 16, 4 up to 32.
constexpr int FM_BK = 128;                  // k per stage: one 128-byte code row
constexpr int FM_UMMA_K = 32;
constexpr int FM_ROW = 128;                 // bytes per staged row (codes and planes)
constexpr int FM_ROWS_PER_TOKEN = 4;        // hi, lo, lo2, zero
constexpr int FM_MAX_STAGES = 8;
constexpr int FM_ACC_BUFS = 2;
constexpr int FM_TMEM_COLS = 512;
constexpr int FM_MAX_CLUSTER = kSkinnyMaxCluster;
constexpr int FM_RED_PITCH = SK_BN + 4;     // floats per token row of a reduction buffer
constexpr int FM_NUM_BARS = 3 * FM_MAX_STAGES + 2 * FM_ACC_BUFS + 2;
constexpr int FM_BAR_BYTES = FM_NUM_BARS * 8 + 16 + 4 * 32;  // + TMEM slot, token exponents
constexpr int FM_SMEM_MAX = 232448;
constexpr int FM_TILE_HDR = 256;            // bytes at the end of the ring for a Tile
static_assert(sizeof(Tile) <= FM_TILE_HDR, "a Tile fits its slot");
static_assert(kF8MmaMaxTokens * FM_ROWS_PER_TOKEN <= 128, "token planes fill the 128 A rows");

struct FmParams {
  CUtensorMap tmW16[TP_MAX_TP];  // codes of W_i: box {128 bytes, 16 rows}, 128-byte swizzle
  CUtensorMap tmW64[TP_MAX_TP];  // box {128 bytes, 64 rows}
  const __nv_bfloat16* X;        // column: X; row: X_i = X + i * x_shard_off
  int64_t ldx, x_shard_off;
  int64_t K;                     // valid k per shard (row) or in all (column)
  const float* bias[TP_MAX_TP];
  const float* wscale[TP_MAX_TP];
  void* Y;
  unsigned int* err;
  int64_t ldy;
  int64_t y_extent;              // elements of Y this call may write (checked builds)
  int64_t fo[TP_MAX_TP + 1];     // column: shard i owns features [fo[i], fo[i+1])
  int64_t yoff[TP_MAX_TP];       // column: element offset of shard i's outputs in Y
  int64_t M, feat_total;
  int tp, row, act, ydt;
  int stages;
  int a_stage_bytes;             // token-plane rows x 128 bytes
  int w_stage_bytes;             // code rows of a B tile x 128 bytes
  int tile_cap;
  int acc_stride, acc_bufs;
  int kb_per_shard, kb_total;
  int cs;
  int ring_bytes;
  int sbuf_floats;               // per-row scales (+ biases) of one tile, in shared memory
  int dump;                      // finish the last tile from shared memory (see the epilogue)
  int red_off;                   // byte offset of the row side's reduction buffer in the ring
};

__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float2 e4m3x2_value(uint32_t c) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)c, __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Split two scaled token values into their three e4m3 planes (exact; see the
// file comment).  Returns the code pairs of hi, lo and lo2.
__device__ __forceinline__ void split_planes(float u0, float u1, uint32_t& hi, uint32_t& lo,
                                             uint32_t& lo2) {
  hi = e4m3x2(u0, u1);
  const float2 h = e4m3x2_value(hi);
  const float r0 = (u0 - h.x) * 16.0f, r1 = (u1 - h.y) * 16.0f;
  lo = e4m3x2(r0, r1);
  const float2 l = e4m3x2_value(lo);
  lo2 = e4m3x2((r0 - l.x) * 16.0f, (r1 - l.y) * 16.0f);
}

// The four lanes 4t .. 4t+3 of token t hold its planes (weighted 1, 1/16,
// 1/256, 0) of the same 16 accumulator columns.  Reduce-scatter them in two
// shuffle steps: afterwards lane 4t+p holds the combined value of 4 of the
// columns, (hi + lo/16) + (lo2/256 + 0) for each, in the same order in every
// lane.  Lane p's columns start at col4(p).  All register indices are static.
__device__ __forceinline__ int col4(int p) { return ((p & 1) << 3) | ((p & 2) << 1); }
__device__ __forceinline__ void combine_planes(const float (&v)[16], int p, float (&out)[4]) {
  const bool b0 = p & 1, b1 = p & 2;
  float h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // step 1 (partner p ^ 1): keep columns [8 b0, 8 b0 + 8), send the others
    const float keep = b0 ? v[8 + i] : v[i];
    const float send = b0 ? v[i] : v[8 + i];
    h[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // step 2 (partner p ^ 2): keep the first or the last 4 of those 8
    const float keep = b1 ? h[4 + i] : h[i];
    const float send = b1 ? h[i] : h[4 + i];
    const float other = __shfl_xor_sync(0xffffffffu, send, 2);
    out[i] = b1 ? other + keep : keep + other;  // (hi + lo/16) + (lo2/256 + 0) everywhere
  }
}

// Barrier of the four epilogue warps only (named barrier 1).
__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// v * 2^e, exactly: a multiply by the power of two when it is a normal float.
__device__ __forceinline__ float scale_pow2(float v, int e) {
  if (e >= -126 && e <= 127) return v * __int_as_float((127 + e) << 23);
  return ldexpf(v, e);
}

// Token scale exponent e: the largest |x| of the token times 2^-e lies in
// [128, 256) (0 for an all-zero token).
__device__ __forceinline__ int token_exponent(float amax) {
  if (!(amax > 0.0f)) return 0;
  int E;
  frexpf(amax, &E);  // amax = m * 2^E, m in [0.5, 1)
  return E - 8;
}

template <int CT>
__global__ void __launch_bounds__(FM_THREADS, 1) f8mma_kernel(const __grid_constant__ FmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  uint8_t* sA = smem;                                       // S plane stages
  uint8_t* sW = smem + (size_t)S * p.a_stage_bytes;         // S code stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(sW + (size_t)S * p.w_stage_bytes);
  uint64_t* full = bars;                        // codes landed
  uint64_t* afull = bars + FM_MAX_STAGES;       // planes written
  uint64_t* empty = bars + 2 * FM_MAX_STAGES;   // both consumed by the MMAs
  uint64_t* tfull = bars + 3 * FM_MAX_STAGES;
  uint64_t* tempty = tfull + FM_ACC_BUFS;
  uint64_t* drain = tempty + FM_ACC_BUFS;
  uint64_t* sready = drain + 1;                 // token exponents written
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + FM_NUM_BARS);
  int* sexp = reinterpret_cast<int*>(bars + FM_NUM_BARS) + 4;  // 32 token exponents
  // one tile's weight-row scales at the tile's row positions (and, with a
  // bias, the biases after them), staged by the epilogue while the MMAs run
  float* sscale = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + FM_BAR_BYTES);
  // After the CTA's last K loop the ring is free.  In dump mode its start
  // holds the raw accumulator rows of the token lanes, dmp[row][nrows + 4]
  // (fp32); the row side's reduction buffer red[token][FM_RED_PITCH] (fp32)
  // follows at red_off.
  float* dmp = reinterpret_cast<float*>(smem);
  float* red = reinterpret_cast<float*>(smem + p.red_off);
  // dump mode: the last tile's pieces, for the threads that finish it
  Tile* last_tile = reinterpret_cast<Tile*>(smem + p.ring_bytes - FM_TILE_HDR);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool swiglu = (!p.row && p.act == TP_ACT_SWIGLU);
  const int rank = p.row ? (int)cluster_ctarank() : 0;
  const int rshard = p.row ? (int)((int64_t)rank * p.tp / p.cs) : 0;  // row: this CTA's shard
  // The next kernel may start its prologue now.  The converters wait for the
  // kernels before this one before reading X; everything that writes Y comes
  // after them (through the MMAs and the barriers); the producer streams the
  // weight codes from the start.
  pdl_launch_dependents();
  const int a_rows = p.a_stage_bytes / FM_ROW;
  const int slots = a_rows / FM_ROWS_PER_TOKEN;  // token slots written per plane stage

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&afull[s]), FM_CONV_THREADS / 32);  // one arrive per converter warp
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < p.acc_bufs; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), 4);  // one arrive per epilogue warp
    }
    mbar_init(smem_u32(drain), 1);
    mbar_init(smem_u32(sready), FM_CONV_THREADS / 32);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.tp; ++i) {
      prefetch_tmap(&p.tmW16[i]);
      prefetch_tmap(&p.tmW64[i]);
    }
  }
  if (warp == 1) tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), FM_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int64_t f0 = 0, f1 = 0;
  if (!p.row) column_range(p, f0, f1);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    const uint64_t pol_w = l2_policy_evict_first();  // the codes are read once
    SK_FOR_EACH_TILE(tl, {
      if (ok) {
        int piece = 0, half = 0, r = 0, h = 0;
        const bool has_box = lane > 0 && tile_box(tl, swiglu, lane - 1, piece, half, r, h);
        int64_t wrow = 0;
        uint32_t woff = 0;
        int wshard = 0;
        if (has_box) {
          const Piece& pc = tl.pc[piece];
          wrow = (swiglu ? (pc.loc / G) * 2 * G + pc.loc % G + half * G : pc.loc) + r;
          woff = (uint32_t)(pc.slot + half * tl.rows + r) * FM_ROW;
          wshard = pc.shard;
        }
        const bool mine = has_box && TP_CHECK(p.err, woff + (uint32_t)h * FM_ROW <=
                                                         (uint32_t)p.w_stage_bytes);
        uint32_t wbytes = 0;
        if (lane == 0) {
          for (int b = 0; b < tl.boxes; ++b) {
            int pi, hf, rr, hh;
            if (tile_box(tl, swiglu, b, pi, hf, rr, hh)) wbytes += (uint32_t)hh * FM_ROW;
          }
        }
        const int nkb = tl.kb1 - tl.kb0;
        const int rot = kb_rotation(nkb, p.row);
        for (int i = 0; i < nkb; ++i) {
          const int kb = kb_at(tl.kb0, nkb, rot, i);
          const int rsh = p.row ? kb / p.kb_per_shard : 0;
          const int kk = p.row ? kb - rsh * p.kb_per_shard : kb;
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
            mbar_arrive_expect_tx(fb, wbytes);
          } else if (mine) {
            const int sh = p.row ? rsh : wshard;
            const CUtensorMap* map = (h == 64) ? &p.tmW64[sh] : &p.tmW16[sh];
            tma_load_2d_hint(smem_u32(sW + (size_t)stage * p.w_stage_bytes) + woff, map,
                             kk * FM_BK, (int)wrow, fb, pol_w);
          }
          __syncwarp();
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    });
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    SK_FOR_EACH_TILE(tl, {
      if (ok && !mbar_wait_bounded(smem_u32(&tempty[acc]), acc_phase ^ 1u)) {
        report_error(p.err, kErrTimeoutMma);
        ok = false;
      }
      if (ok) {
        tc_fence_after();
        const int nrows = swiglu ? 2 * tl.rows : tl.rows;
        const int n0 = nrows < SK_BN ? nrows : SK_BN;
        const int n1 = nrows - n0;
        const uint32_t idesc0 = idesc_e4m3_f32(128, n0);
        const uint32_t idesc1 = idesc_e4m3_f32(128, n1 > 0 ? n1 : 16);
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * p.acc_stride);
        if (!TP_CHECK(p.err, nrows * FM_ROW <= p.w_stage_bytes &&
                                 acc * p.acc_stride + nrows <= FM_TMEM_COLS))
          ok = false;
        for (int i = 0; ok && i < tl.kb1 - tl.kb0; ++i) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase) ||
              !mbar_wait_bounded(smem_u32(&afull[stage]), phase)) {
            report_error(p.err, kErrTimeoutMma);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_sw128(smem_u32(sA + (size_t)stage * p.a_stage_bytes));
          const uint32_t wbase = smem_u32(sW + (size_t)stage * p.w_stage_bytes);
          const uint64_t bdesc0 = sdesc_sw128(wbase);
          const uint64_t bdesc1 = sdesc_sw128(wbase + SK_BN * FM_ROW);
#pragma unroll
          for (int k = 0; k < FM_BK / FM_UMMA_K; ++k) {
            // K = 32 codes = 32 bytes: the start address advances by 2 x 16 bytes
            const uint32_t accum = (i > 0 || k > 0) ? 1u : 0u;
            mma_e4m3(d_tmem, adesc + (uint64_t)(k * 2), bdesc0 + (uint64_t)(k * 2), idesc0, accum);
            if (n1 > 0)
              mma_e4m3(d_tmem + SK_BN, adesc + (uint64_t)(k * 2), bdesc1 + (uint64_t)(k * 2),
                       idesc1, accum);
          }
          mma_commit(smem_u32(&empty[stage]));  // codes and planes reusable once these finish
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) mma_commit(smem_u32(&tfull[acc]));
      }
      if (++acc == p.acc_bufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    });
    mma_commit(smem_u32(drain));
    if (!mbar_wait_bounded(smem_u32(drain), 0)) report_error(p.err, kErrTimeoutDrain);
  } else if (warp >= FM_EPI_WARP0 && warp < FM_EPI_WARP0 + 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                // TMEM lane quadrant this warp may access
    const int tok = q * 8 + (lane >> 2);   // this lane's token
    const int plane = lane & 3;            // and plane (3: the zero row)
    const bool has_tokens = q * 8 < p.M;   // warp-uniform
    const bool live = tok < p.M;
    // planes are weighted 1, 1/16, 1/256 (the zero row 0) before the butterfly
    const float pw = plane == 0 ? 1.0f : plane == 1 ? 0.0625f : plane == 2 ? 0.00390625f : 0.0f;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = mbar_wait_bounded(smem_u32(sready), 0);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) report_error(p.err, kErrTimeoutEpilogue);
    const int e = live ? sexp[tok] : 0;
    const int et = threadIdx.x - FM_EPI_WARP0 * 32;  // 0 .. 127
    SK_FOR_EACH_TILE(tl, {
      // Stage the tile's scales (and biases): row r of the B tile (gate rows,
      // then the up rows at the same slots) -> sscale[r]; biases at
      // sscale[nrows + r].  The barriers keep the previous tile's readers and
      // this tile's writers apart.
      const int nrows = swiglu ? 2 * tl.rows : tl.rows;
      const bool has_bias = !swiglu && (p.row ? p.bias[0] != nullptr : true);
      epi_bar_sync();
      for (int r = et; r < nrows; r += 128) {
        const int rr = r < tl.rows ? r : r - tl.rows;  // slot row
        const int half = r < tl.rows ? 0 : 1;          // SwiGLU: 0 gate, 1 up
        float scv = 0.0f, bv = 0.0f;
        for (int i = 0; i < tl.n; ++i) {
          const Piece& pc = tl.pc[i];
          const int j = rr - pc.slot;
          if (j < 0 || j >= pc.c) continue;
          const int sh = p.row ? rshard : pc.shard;
          const int64_t wr = swiglu ? (pc.loc / G) * 2 * G + pc.loc % G + half * G + j : pc.loc + j;
          scv = __ldg(p.wscale[sh] + wr);
          const float* b = p.row ? p.bias[0] : p.bias[pc.shard];
          if (has_bias && b) bv = __ldg(b + pc.loc + j);
        }
        if (TP_CHECK(p.err, r < p.sbuf_floats && (!has_bias || nrows + r < p.sbuf_floats))) {
          sscale[r] = scv;
          if (has_bias) sscale[nrows + r] = bv;
        }
      }
      epi_bar_sync();
      if (ok) {
        ok = mbar_wait_bounded(smem_u32(&tfull[acc]), acc_phase);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && lane == 0) report_error(p.err, kErrTimeoutEpilogue);
      }
      if (ok) {
        tc_fence_after();
        const uint32_t taddr =
            tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.acc_stride);
        const int drow = q * 32 + lane;  // this lane's accumulator row
        if (p.dump && tile_is_last) {
          if (et == 0) *last_tile = tl;
          // Dump mode: copy the token lanes' raw accumulators to dmp; all
          // eight epilogue and converter warps finish them below.  (With
          // few tokens only one or two warps hold token lanes, and the
          // activation and stores would run on them alone.)
          if (has_tokens) {
            const int pitch = nrows + 4;
#pragma unroll 1
            for (int c0 = 0; c0 < nrows;) {
              float v[32];
              const int w = nrows - c0 >= 32 ? 32 : 16;
              if (w == 32) {
                tmem_ld32(taddr + (uint32_t)c0, v);
              } else {
                float v16[16];
                tmem_ld16(taddr + (uint32_t)c0, v16);
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = v16[j];
              }
              if (drow < 4 * p.M &&
                  TP_CHECK(p.err, (int64_t)(drow * pitch + c0 + w) * 4 <= p.red_off)) {
                float4* d = reinterpret_cast<float4*>(dmp + drow * pitch + c0);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  if (4 * j < w) d[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
              }
              c0 += w;
            }
          }
        } else if (has_tokens && p.row && p.cs > 1) {
          // 16 columns per step; combine_planes leaves lane `plane` of a token
          // with the combined values of columns col4(plane) .. col4(plane) + 3
          const int c = tl.pc[0].c;
#pragma unroll 1
          for (int j0 = 0; j0 < c; j0 += 16) {
            float v[16], w[4];
            tmem_ld16(taddr + (uint32_t)j0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] *= pw;
            combine_planes(v, plane, w);
            const int col = j0 + col4(plane);
            if (live && col < c &&
                TP_CHECK(p.err, (int64_t)(tok * FM_RED_PITCH + col + 4) * 4 <= p.ring_bytes)) {
              // this CTA's partial belongs to shard rshard: its row scales
#pragma unroll
              for (int j = 0; j < 4; ++j)
                w[j] = (col + j < c) ? sscale[col + j] * scale_pow2(w[j], e) : 0.0f;
              *reinterpret_cast<float4*>(red + tok * FM_RED_PITCH + col) =
                  make_float4(w[0], w[1], w[2], w[3]);
            }
          }
        } else if (has_tokens) {
          for (int i = 0; i < tl.n; ++i) {
            const Piece& pc = tl.pc[i];
            const int64_t base = (p.row ? 0 : p.yoff[pc.shard]) + (int64_t)tok * p.ldy;
            const bool bias = has_bias && (p.row ? p.bias[0] : p.bias[pc.shard]) != nullptr;
            // Finish 16 columns [j0, j0 + 16): weight the planes, combine them,
            // scale, activate, store this lane's 4 of them.
            auto finish16 = [&](const float* vin, const float* uin, int j0) {
              float v[16], u[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                v[j] = vin[j] * pw;
                u[j] = swiglu ? uin[j] * pw : 0.0f;
              }
              float g4[4], u4[4];
              combine_planes(v, plane, g4);
              if (swiglu) combine_planes(u, plane, u4);
              const int col = j0 + col4(plane);  // this lane's 4 columns
              const int valid = pc.c - col < 4 ? pc.c - col : 4;
              if (!live || valid <= 0) return;
              float w[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                if (j >= valid) {
                  w[j] = 0.0f;
                  continue;
                }
                const int r = pc.slot + col + j;  // B tile row of this output (gate row)
                float z = sscale[r] * scale_pow2(g4[j], e);
                if (swiglu) {
                  const float up = sscale[tl.rows + r] * scale_pow2(u4[j], e);
                  z = act_silu(z) * up;
                } else {
                  if (bias) z += sscale[nrows + r];
                  if (!p.row && p.act == TP_ACT_GELU_ERF) z = act_gelu_erf(z);
                }
                w[j] = z;
              }
              if (TP_CHECK(p.err, base + pc.loc + col + valid <= p.y_extent))
                store_row4(p.Y, p.ydt, base, pc.loc + col, valid, w);
            };
            // 32 columns per TMEM wait while they stay inside the piece's slot
            // (slots are multiples of 16 wide), then 16
            const int slot_cols = (pc.c + 15) / 16 * 16;
#pragma unroll 1
            for (int j0 = 0; j0 < pc.c;) {
              const uint32_t tg = taddr + (uint32_t)(pc.slot + j0);
              const uint32_t tu = taddr + (uint32_t)(tl.rows + pc.slot + j0);
              if (slot_cols - j0 >= 32) {
                float v[32], u[32];
                if (swiglu)
                  tmem_ld32x2(tg, tu, v, u);
                else
                  tmem_ld32(tg, v);
                finish16(v, u, j0);
                finish16(v + 16, u + 16, j0 + 16);
                j0 += 32;
              } else {
                float v[16], u[16];
                if (swiglu)
                  tmem_ld16x2(tg, tu, v, u);
                else
                  tmem_ld16(tg, v);
                finish16(v, u, j0);
                j0 += 16;
              }
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
  } else if (warp >= FM_CONV_WARP0) {
    // ------------------------------------------------------------ converters
    const int cw = warp - FM_CONV_WARP0;
    const int ct = threadIdx.x - FM_CONV_WARP0 * 32;
    pdl_wait();  // X may be the output of the kernel before this one
    // Token scales over this CTA's k-range: the column side's is all of K;
    // the row side's lies inside shard rshard.
    int64_t kr0 = 0, kr1 = p.K;
    const __nv_bfloat16* xbase = p.X;
    if (p.row) {
      const Tile tl = row_tile(p, rank);
      const int sh = tl.kb0 / p.kb_per_shard;
      xbase = p.X + (int64_t)sh * p.x_shard_off;
      kr0 = (int64_t)(tl.kb0 - sh * p.kb_per_shard) * FM_BK;
      kr1 = imin((int64_t)(tl.kb1 - sh * p.kb_per_shard) * FM_BK, p.K);
    }
    for (int t = cw; t < p.M; t += FM_CONV_THREADS / 32) {
      const __nv_bfloat16* xr = xbase + (int64_t)t * p.ldx;
      float m = 0.0f;
      for (int64_t k = kr0 + 8 * lane; k < kr1; k += 8 * 32) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + k));
        float f[8];
        unpack_bf16x8(v, f);
#pragma unroll
        for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) sexp[t] = token_exponent(m);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(sready));
    bool ok = mbar_wait_bounded(smem_u32(sready), 0);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) report_error(p.err, kErrTimeoutConvert);
    // Per k-block, task = (token slot, 8 of the block's 128 k): its 8 k of the
    // three planes go to rows 4t .. 4t+2 and zeros to row 4t+3, 8 bytes each
    // at byte (c ^ (row mod 8)) * 16 + 8 * half of the row, c = the 16-byte
    // chunk (the 128-byte swizzle).  A thread's tasks are ct, ct + 128, ...;
    // the X values of a k-block are loaded two k-blocks ahead of its
    // conversion, so the L2 latency of X overlaps the conversions between.
    const int ntasks = slots * 16;
    int stage = 0;
    uint32_t phase = 0;
    SK_FOR_EACH_TILE(tl, {
      uint4 x0[CT], x1[CT], x2[CT];
      auto load_x = [&](int kb, uint4 (&dst)[CT]) {
        const int rsh = p.row ? kb / p.kb_per_shard : 0;
        const int kk = p.row ? kb - rsh * p.kb_per_shard : kb;
        const __nv_bfloat16* xs = p.X + (int64_t)rsh * p.x_shard_off;
#pragma unroll
        for (int i = 0; i < CT; ++i) {
          const int task = ct + i * FM_CONV_THREADS;
          const int t = task >> 4;
          const int64_t k0 = (int64_t)kk * FM_BK + 8 * (task & 15);
          dst[i] = make_uint4(0, 0, 0, 0);
          if (kb < tl.kb1 && task < ntasks && t < p.M && k0 < p.K)
            dst[i] = __ldg(reinterpret_cast<const uint4*>(xs + (int64_t)t * p.ldx + k0));
        }
      };
      // One k-block: wait for its stage to be free, convert, release it to
      // the MMA.  (A buffer loaded for a later k-block is never copied
      // before its use: a copy would wait for the load.)
      auto convert = [&](const uint4 (&x)[CT]) {
        bool got = true;
        if (lane == 0) got = mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u);
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          if (lane == 0) report_error(p.err, kErrTimeoutConvert);
          ok = false;
          return;
        }
        uint8_t* dst = sA + (size_t)stage * p.a_stage_bytes;
#pragma unroll
        for (int i = 0; i < CT; ++i) {
          const int task = ct + i * FM_CONV_THREADS;
          if (task >= ntasks) break;
          const int t = task >> 4, c = (task & 15) >> 1, half = task & 1;
          uint2 qh = make_uint2(0, 0), ql = qh, ql2 = qh;
          if (t < p.M) {
            float f[8];
            unpack_bf16x8(x[i], f);
            // u = x * 2^-e, exactly: a multiply by the power of two when it is
            // a normal float, else ldexpf
            const int e = sexp[t];
            if (e >= -126 && e <= 126) {
              const float sc = __int_as_float((127 - e) << 23);
#pragma unroll
              for (int j = 0; j < 8; ++j) f[j] *= sc;
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) f[j] = ldexpf(f[j], -e);
            }
            uint32_t h[4], l[4], l2[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) split_planes(f[2 * j], f[2 * j + 1], h[j], l[j], l2[j]);
            qh = make_uint2(h[0] | h[1] << 16, h[2] | h[3] << 16);
            ql = make_uint2(l[0] | l[1] << 16, l[2] | l[3] << 16);
            ql2 = make_uint2(l2[0] | l2[1] << 16, l2[2] | l2[3] << 16);
          }
          const int r0 = FM_ROWS_PER_TOKEN * t;
          if (TP_CHECK(p.err, (r0 + 4) * FM_ROW <= p.a_stage_bytes)) {
            const int cb = 8 * half;
            *reinterpret_cast<uint2*>(dst + (r0 + 0) * FM_ROW + ((c ^ ((r0 + 0) & 7)) << 4) + cb) = qh;
            *reinterpret_cast<uint2*>(dst + (r0 + 1) * FM_ROW + ((c ^ ((r0 + 1) & 7)) << 4) + cb) = ql;
            *reinterpret_cast<uint2*>(dst + (r0 + 2) * FM_ROW + ((c ^ ((r0 + 2) & 7)) << 4) + cb) = ql2;
            *reinterpret_cast<uint2*>(dst + (r0 + 3) * FM_ROW + ((c ^ ((r0 + 3) & 7)) << 4) + cb) =
                make_uint2(0, 0);
          }
        }
        fence_proxy_async_smem();  // the MMA reads these writes through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&afull[stage]));
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      };
      // the K loop in the producer's rotated order
      const int nkb = tl.kb1 - tl.kb0;
      const int rot = kb_rotation(nkb, p.row);
      if (ok) {
        load_x(kb_at(tl.kb0, nkb, rot, 0), x0);
        load_x(kb_at(tl.kb0, nkb, rot, 1), x1);
      }
      for (int i = 0; ok && i < nkb; i += 3) {
        load_x(kb_at(tl.kb0, nkb, rot, i + 2), x2);
        convert(x0);
        if (!ok || i + 1 >= nkb) break;
        load_x(kb_at(tl.kb0, nkb, rot, i + 3), x0);
        convert(x1);
        if (!ok || i + 2 >= nkb) break;
        load_x(kb_at(tl.kb0, nkb, rot, i + 4), x1);
        convert(x2);
      }
    });
  }

  if (p.dump && warp >= FM_EPI_WARP0) {
    // ------------------------------------------------------------ dump-mode finish
    // The epilogue warps have copied the last tile's token lanes to dmp (the
    // converters arrive here after their K loop).  256 threads then take a
    // tile row each, for every token: planes combined as (hi + lo/16) + lo2/256,
    // times 2^e and the row's scale (staged in sscale), then the bias and
    // activation, and the store (row side with a cluster: the partial goes
    // to red for the cluster's sum).
    asm volatile("bar.sync 2, 256;" ::: "memory");
    const int bt = threadIdx.x - FM_EPI_WARP0 * 32;
    const Tile& tl = *last_tile;  // written before the barrier by the epilogue
    const int nrows = swiglu ? 2 * tl.rows : tl.rows;
    const int pitch = nrows + 4;
    const bool has_bias = !swiglu && (p.row ? p.bias[0] != nullptr : true);
    // thread bt takes tile rows bt, bt + 256, ... and every token of each
    for (int r = bt; r < tl.rows; r += 256) {
      int pi = -1;
      for (int i = 0; i < tl.n; ++i)
        if (r >= tl.pc[i].slot && r < tl.pc[i].slot + tl.pc[i].c) pi = i;
      if (pi < 0) continue;  // a padding row of a slot
      const int shard = tl.pc[pi].shard;
      const int64_t col = tl.pc[pi].loc + (r - tl.pc[pi].slot);  // shard-local output
      const float sg = sscale[r];
      const float su = swiglu ? sscale[tl.rows + r] : 0.0f;
      const float* b = p.row ? p.bias[0] : p.bias[shard];
      const float bv = (has_bias && b) ? sscale[nrows + r] : 0.0f;
      const int64_t obase = (p.row ? 0 : p.yoff[shard]) + col;
      for (int t = 0; t < p.M; ++t) {
        const int e = sexp[t];
        const float* d0 = dmp + (4 * t) * pitch;
        float z = sg * scale_pow2((d0[r] + d0[pitch + r] * 0.0625f) + d0[2 * pitch + r] * 0.00390625f, e);
        if (p.row && p.cs > 1) {
          if (TP_CHECK(p.err, (int64_t)(p.red_off / 4) + t * FM_RED_PITCH + r < p.ring_bytes / 4))
            red[t * FM_RED_PITCH + r] = z;
          continue;
        }
        if (swiglu) {
          const int ru = tl.rows + r;
          const float up =
              su * scale_pow2((d0[ru] + d0[pitch + ru] * 0.0625f) + d0[2 * pitch + ru] * 0.00390625f, e);
          z = act_silu(z) * up;
        } else {
          z += bv;
          if (!p.row && p.act == TP_ACT_GELU_ERF) z = act_gelu_erf(z);
        }
        const int64_t o = obase + (int64_t)t * p.ldy;
        if (TP_CHECK(p.err, o < p.y_extent)) store_out(p.Y, p.ydt, o, z);
      }
    }
  }

  __syncthreads();
  if (p.row && p.cs > 1) {
    // ---------------------------------------------------------- cluster reduction
    // Every thread of every CTA of the cluster passes both barriers.
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
        const int64_t tk = it / span;
        const int j = j_lo + (int)(it - tk * span);
        const uint32_t off = (uint32_t)((tk * FM_RED_PITCH + j) * 4);
        float sum = 0.0f;
        for (int r = 0; r < p.cs; ++r) sum += dsmem_ld_f32(dsmem_addr(red_s + off, (uint32_t)r));
        if (bias) sum += __ldg(bias + loc + j);
        if (TP_CHECK(p.err, tk * p.ldy + loc + j < p.y_extent))
          store_out(p.Y, p.ydt, tk * p.ldy + loc + j, sum);
      }
    }
    cluster_sync_all();  // no CTA leaves while a peer still reads its buffer
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, FM_TMEM_COLS);
  }
}

}  // namespace

tp_status prepare_f8mma(const LinearProblem& p, Launch* L) {
  if (!p.fp8 || p.xdt != TP_BF16 || p.M < 1 || p.M > kF8MmaMaxTokens) return TP_ERR_UNSUPPORTED;
  if (p.row && p.tp > FM_MAX_CLUSTER) return TP_ERR_UNSUPPORTED;
  FmParams fp{};
  fp.err = device_error_word();
  if (!fp.err) return TP_ERR_CUDA;
  for (int i = 0; i < p.tp; ++i) {
    const uint64_t rows = (uint64_t)(p.row ? p.w_rows : p.wr[i]);
    if (!make_tma_map_u8(&fp.tmW16[i], p.W[i], (uint64_t)p.K, rows, (uint64_t)p.K, FM_ROW, 16,
                         true) ||
        !make_tma_map_u8(&fp.tmW64[i], p.W[i], (uint64_t)p.K, rows, (uint64_t)p.K, FM_ROW, 64,
                         true))
      return TP_ERR_CUDA;
  }
  fp.X = static_cast<const __nv_bfloat16*>(p.X);
  fp.ldx = p.ldx;
  fp.x_shard_off = p.x_shard_off;
  fp.K = p.K;
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
  fp.kb_per_shard = (int)((p.K + FM_BK - 1) / FM_BK);
  fp.kb_total = fp.kb_per_shard * (p.row ? p.tp : 1);

  const int sms = sm_count();
  int grid = 1;
  fp.cs = 1;
  const bool swiglu = !p.row && p.act == TP_ACT_SWIGLU;
  int tile_rows = SK_BN;
  if (p.row) {
    // tiles of bn outputs; tp x j CTAs per cluster, each inside one shard
    int resident[FM_MAX_CLUSTER + 1];
    resident_clusters(reinterpret_cast<const void*>(f8mma_kernel<1>), FM_THREADS, FM_SMEM_MAX,
                      FM_MAX_CLUSTER, p.tp, resident);
    const RowTiling rt = choose_row_tiling(p.n_out, fp.kb_total, fp.kb_per_shard, sms,
                                           FM_MAX_CLUSTER, p.tp, resident);
    if (rt.tiles * rt.cs > INT32_MAX) return TP_ERR_BAD_SHAPE;
    fp.cs = rt.cs;
    grid = (int)(rt.tiles * rt.cs);
    fp.tile_cap = rt.bn;
    tile_rows = rt.bn;
  } else {
    const int64_t units = (fp.feat_total + SK_GRAIN - 1) / SK_GRAIN;
    grid = (int)std::max<int64_t>(1, std::min<int64_t>(units, sms));
    const int64_t max_range = (units + grid - 1) / grid * SK_GRAIN;
    fp.tile_cap = (int)std::min<int64_t>(SK_BN, max_range);
    tile_rows = swiglu ? 2 * fp.tile_cap : fp.tile_cap;
  }
  // plane stage: 4 rows per token, whole 8-row swizzle atoms
  const int a_rows = (int)((FM_ROWS_PER_TOKEN * p.M + 7) / 8 * 8);
  fp.a_stage_bytes = a_rows * FM_ROW;
  fp.w_stage_bytes = tile_rows * FM_ROW;
  fp.acc_stride = (tile_rows + 31) / 32 * 32;
  fp.acc_bufs = (FM_ACC_BUFS * fp.acc_stride <= FM_TMEM_COLS) ? FM_ACC_BUFS : 1;
  // scales of one tile's rows, plus as many biases when the call has a bias
  // (non-SwiGLU column calls take their biases from there, a row call with
  // one cluster CTA per tile too)
  fp.sbuf_floats = 2 * tile_rows;
  if (swiglu) fp.sbuf_floats = tile_rows;
  const int avail = FM_SMEM_MAX - 1024 - FM_BAR_BYTES - 4 * fp.sbuf_floats;
  const int per_stage = fp.a_stage_bytes + fp.w_stage_bytes;
  const int stages = std::min(FM_MAX_STAGES, avail / per_stage);
  if (stages < 2) return TP_ERR_UNSUPPORTED;
  fp.stages = stages;
  const int ring = stages * per_stage;
  fp.ring_bytes = ring;
  // The MMA reads a full 128-row A tile from each plane stage: the rows past
  // the last plane stage are code stages, which must be there.  The row
  // side's reduction buffer reuses the ring.
  if ((stages - 1) * fp.a_stage_bytes + 128 * FM_ROW > ring) return TP_ERR_UNSUPPORTED;
  if (p.row && fp.cs > 1 && (int64_t)p.M * FM_RED_PITCH * 4 > ring) return TP_ERR_UNSUPPORTED;
  // Dump mode when the token lanes' raw accumulators of a tile (4 rows per
  // token, tile_rows + 4 floats each) and the reduction buffer fit the ring
  // together.
  const int64_t dump_bytes = (int64_t)FM_ROWS_PER_TOKEN * p.M * (tile_rows + 4) * 4;
  const int64_t red_bytes = (p.row && fp.cs > 1) ? (int64_t)p.M * FM_RED_PITCH * 4 : 0;
  fp.dump = (dump_bytes + red_bytes + FM_TILE_HDR <= ring) ? 1 : 0;
  fp.red_off = fp.dump ? (int)dump_bytes : 0;
  const int smem = 1024 + ring + FM_BAR_BYTES + 4 * fp.sbuf_floats;

  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    for (const void* k : {reinterpret_cast<const void*>(f8mma_kernel<1>),
                          reinterpret_cast<const void*>(f8mma_kernel<2>),
                          reinterpret_cast<const void*>(f8mma_kernel<4>)})
      if (attr_err == cudaSuccess)
        attr_err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        FM_SMEM_MAX);
  });
  if (attr_err != cudaSuccess) return TP_ERR_CUDA;
  // conversion tasks per converter thread: 16 per token slot over 128 threads
  const int slots = a_rows / FM_ROWS_PER_TOKEN;
  const int ct = (slots * 16 + FM_CONV_THREADS - 1) / FM_CONV_THREADS;
  L->kernel = ct <= 1   ? reinterpret_cast<const void*>(f8mma_kernel<1>)
              : ct <= 2 ? reinterpret_cast<const void*>(f8mma_kernel<2>)
                        : reinterpret_cast<const void*>(f8mma_kernel<4>);
  L->grid = dim3((unsigned)grid);
  L->block = dim3(FM_THREADS);
  L->smem = (size_t)smem;
  L->cluster = (unsigned)fp.cs;
  L->pdl = true;
  L->set_params(fp);
  return TP_OK;
}

}  // namespace tpla
