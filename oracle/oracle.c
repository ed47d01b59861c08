/*
 * oracle.c -- plain, slow fp64 CPU oracle for the tensor-parallel split of a
 * transformer layer's linear algebra.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA path.
 *
 * Conventions
 *   - Weights are stored like nn.Linear: W is [out_features, in_features],
 *     row-major, so y = x . W^T + b.
 *   - Every input arrives as float: bf16 and fp32 values widen to fp32
 *     exactly, so the oracle sees the very bits the GPU sees.  All arithmetic
 *     is fp64; outputs are fp64.
 *   - Dot products run k = 0 .. K-1 in order, one fp64 accumulator.  No
 *     blocking, no reordering.
 *   - Parallelism (OpenMP) is over independent output elements only.
 *
 * Sources (page title -- section):
 *   [P3] "Understanding Tensor Parallelism for Multi-GPU LLM Serving" --
 *        "How Tensor Parallelism Works Under the Hood" (column and row
 *        parallelism, the FFN pairing) and "Implementing Tensor Parallelism
 *        with Hugging Face Accelerate" (ColumnParallelLinear /
 *        RowParallelLinear: shard shapes, divisibility asserts, bias added once
 *        after the all-reduce, F.gelu between the two layers).
 *   [P4] "What is tensor parallelism?" -- "How a layer is split" (heads go to
 *        different GPUs) and "Why it helps when serving" (tp must divide the
 *        head count).
 *   [P5] "Tensor parallel serving" -- "Simulating the split, and proving it is
 *        correct" (row slices W[:split], W[split:], concatenation) and
 *        "Column-parallel and row-parallel layers, paired" (sum, not concat).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - GELU is the exact erf form, the default of torch.nn.functional.gelu that
 *     [P3]'s FFN demo calls.
 *   - SwiGLU is silu(x.Wg^T) * (x.Wu^T), silu(z) = z / (1 + e^-z); gate and up
 *     use the same column split; no bias.  (No page defines it; the
 *     Llama-2-70B-shaped workloads use it.)
 *   - The row-parallel input of shard i is the shard-local column output h_i
 *     ([P3]'s forward re-slices an already-sharded input, which cannot run for
 *     rank >= 1; the pairing described in [P3] and [P5] feeds h_i directly).
 *   - Row partials are summed in shard order 0..p-1, then the bias is added
 *     once.
 *   - The QKV weight stores rows [Q heads 0..H-1 ; K heads 0..Hkv-1 ; V heads
 *     0..Hkv-1], head_dim rows per head.  Shard i takes Q heads
 *     [i*H/p, (i+1)*H/p), K heads and V heads [i*Hkv/p, (i+1)*Hkv/p).
 *   - tp must divide the KV head count too (no KV replication).
 *   - Where the method stores an intermediate in bf16, the oracle rounds it
 *     to bf16 (round to nearest, ties to even) at that point.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
  ORC_OK = 0,
  ORC_ERR_NULL = 1,
  ORC_ERR_NOT_DIVISIBLE = 2,
  ORC_ERR_BAD_SHAPE = 3,
  ORC_ERR_NOMEM = 8
};

enum { ORC_ACT_NONE = 0, ORC_ACT_GELU = 1, ORC_ACT_SWIGLU = 2 };

/* ------------------------------------------------------------------------ */
/* Scalar functions                                                          */
/* ------------------------------------------------------------------------ */

/* GELU, exact form: z * Phi(z) = 0.5 z (1 + erf(z / sqrt 2)). */
double orc_gelu(double z) { return 0.5 * z * (1.0 + erf(z / sqrt(2.0))); }

/* SiLU (swish): z * sigmoid(z). */
double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * Round an fp64 value to the nearest bf16 value (8 significant bits, 8-bit
 * exponent), ties to even, returned as fp64.  bf16 shares fp32's exponent
 * range: normals down to 2^-126, subnormals with quantum 2^-133, overflow to
 * infinity at 2^128 (after rounding).
 */
double orc_round_bf16(double x) {
  if (isnan(x) || isinf(x) || x == 0.0) return x;
  double a = fabs(x);
  double r;
  if (a < ldexp(1.0, -126)) {
    /* subnormal range: fixed quantum 2^-133 */
    r = ldexp(nearbyint(ldexp(a, 133)), -133);
  } else {
    int e;
    double m = frexp(a, &e);          /* a = m * 2^e, m in [0.5, 1) */
    r = ldexp(nearbyint(ldexp(m, 8)), e - 8); /* keep 8 significant bits */
  }
  if (r >= ldexp(1.0, 128)) r = INFINITY;
  return x < 0 ? -r : r;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

static double apply_act(int act, double z) {
  if (act == ORC_ACT_GELU) return orc_gelu(z);
  return z;
}

/* ------------------------------------------------------------------------ */
/* The unsharded layer: the plain definition                                 */
/* ------------------------------------------------------------------------ */

/* One output element: sum_k x[k] * w[k], k in order, fp64. */
static double dot(int64_t K, const float* x, const float* w) {
  double s = 0.0;
  for (int64_t k = 0; k < K; ++k) s += (double)x[k] * (double)w[k];
  return s;
}

/*
 * y = act(x . W^T + b), unsharded.  X [M, K] (row stride ldx), W [N, K]
 * (row stride ldw), b [N] or NULL, Y [M, N] (row stride ldy).
 * act: ORC_ACT_NONE or ORC_ACT_GELU.
 */
int orc_linear(int64_t M, int64_t K, int64_t N, const float* X, int64_t ldx,
               const float* W, int64_t ldw, const float* b, int act, double* Y,
               int64_t ldy) {
  if (M < 0 || K < 0 || N < 0) return ORC_ERR_BAD_SHAPE;
  if ((M * N > 0) && (!X || !W || !Y)) return ORC_ERR_NULL;
  if (act != ORC_ACT_NONE && act != ORC_ACT_GELU) return ORC_ERR_BAD_SHAPE;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double z = dot(K, X + m * ldx, W + n * ldw);
      if (b) z += (double)b[n];
      Y[m * ldy + n] = apply_act(act, z);
    }
  return ORC_OK;
}

/* y = silu(x . Wg^T) * (x . Wu^T), unsharded, no bias. */
int orc_swiglu(int64_t M, int64_t K, int64_t N, const float* X, int64_t ldx,
               const float* Wg, const float* Wu, int64_t ldw, double* Y,
               int64_t ldy) {
  if (M < 0 || K < 0 || N < 0) return ORC_ERR_BAD_SHAPE;
  if ((M * N > 0) && (!X || !Wg || !Wu || !Y)) return ORC_ERR_NULL;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double g = dot(K, X + m * ldx, Wg + n * ldw);
      double u = dot(K, X + m * ldx, Wu + n * ldw);
      Y[m * ldy + n] = orc_silu(g) * u;
    }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* The sharded split, done literally                                         */
/* ------------------------------------------------------------------------ */

/*
 * Column-parallel linear [P3 "How Tensor Parallelism Works Under the Hood";
 * P5 "Simulating the split, and proving it is correct"].
 *
 * Shard i holds rows [i*N/p, (i+1)*N/p) of W (an output slice) and the same
 * slice of b, computes Y_i = act(X . W_i^T + b_i) from the full X, and writes
 * it into column block i of Y: that placement is the concatenation.
 * act = ORC_ACT_SWIGLU takes a second weight Wu split the same way.
 * N % p != 0 is rejected, as the ColumnParallelLinear assert does.
 */
int orc_column_parallel(int tp, int64_t M, int64_t K, int64_t N,
                        const float* X, int64_t ldx, const float* W,
                        const float* Wu, int64_t ldw, const float* b, int act,
                        double* Y, int64_t ldy) {
  if (tp < 1) return ORC_ERR_BAD_SHAPE;
  if (N % tp != 0) return ORC_ERR_NOT_DIVISIBLE;
  int64_t ns = N / tp; /* out_features_per_partition */
  for (int i = 0; i < tp; ++i) {
    const float* Wi = W + (int64_t)i * ns * ldw;
    double* Yi = Y + (int64_t)i * ns; /* column block i of the concatenation */
    int rc;
    if (act == ORC_ACT_SWIGLU) {
      const float* Wui = Wu ? Wu + (int64_t)i * ns * ldw : NULL;
      rc = orc_swiglu(M, K, ns, X, ldx, Wi, Wui, ldw, Yi, ldy);
    } else {
      const float* bi = b ? b + (int64_t)i * ns : NULL;
      rc = orc_linear(M, K, ns, X, ldx, Wi, ldw, bi, act, Yi, ldy);
    }
    if (rc != ORC_OK) return rc;
  }
  return ORC_OK;
}

/*
 * Column-parallel linear with explicit per-shard widths (the uneven split of
 * [P5 "Try it yourself"], e.g. 9 outputs as 5 + 4).  widths[i] > 0 and
 * sum(widths) == N.  act: none or GELU.
 */
int orc_column_parallel_uneven(int tp, const int64_t* widths, int64_t M,
                               int64_t K, int64_t N, const float* X,
                               int64_t ldx, const float* W, int64_t ldw,
                               const float* b, int act, double* Y,
                               int64_t ldy) {
  if (tp < 1 || !widths) return ORC_ERR_BAD_SHAPE;
  int64_t total = 0;
  for (int i = 0; i < tp; ++i) {
    if (widths[i] < 0) return ORC_ERR_BAD_SHAPE;
    total += widths[i];
  }
  if (total != N) return ORC_ERR_BAD_SHAPE;
  int64_t row0 = 0;
  for (int i = 0; i < tp; ++i) {
    int rc = orc_linear(M, K, widths[i], X, ldx, W + row0 * ldw, ldw,
                        b ? b + row0 : NULL, act, Y + row0, ldy);
    if (rc != ORC_OK) return rc;
    row0 += widths[i];
  }
  return ORC_OK;
}

/*
 * Row-parallel linear [P3 "How Tensor Parallelism Works Under the Hood" and
 * RowParallelLinear; P5 "Column-parallel and row-parallel layers, paired"].
 *
 * Shard i holds columns [i*K/p, (i+1)*K/p) of W (an input slice, shape
 * [N, K/p]) and receives the matching columns X_i of the input.  It computes
 * the partial Y_i = X_i . W_i^T.  The all-reduce sums the partials (here in
 * shard order 0..p-1) and the bias is added once, after the sum.
 * K % p != 0 is rejected, as the RowParallelLinear assert does.
 */
int orc_row_parallel(int tp, int64_t M, int64_t K, int64_t N, const float* X,
                     int64_t ldx, const float* W, int64_t ldw, const float* b,
                     double* Y, int64_t ldy) {
  if (tp < 1) return ORC_ERR_BAD_SHAPE;
  if (M < 0 || K < 0 || N < 0) return ORC_ERR_BAD_SHAPE;
  if (K % tp != 0) return ORC_ERR_NOT_DIVISIBLE;
  int64_t ks = K / tp; /* in_features_per_partition */
  double* part = (double*)malloc(sizeof(double) * (size_t)(M * N > 0 ? M * N : 1));
  if (!part) return ORC_ERR_NOMEM;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) Y[m * ldy + n] = 0.0;
  for (int i = 0; i < tp; ++i) {
    /* partial on "device" i */
    int rc = orc_linear(M, ks, N, X + (int64_t)i * ks, ldx,
                        W + (int64_t)i * ks, ldw, NULL, ORC_ACT_NONE, part, N);
    if (rc != ORC_OK) {
      free(part);
      return rc;
    }
    /* all-reduce (sum), accumulated in shard order */
    for (int64_t m = 0; m < M; ++m)
      for (int64_t n = 0; n < N; ++n) Y[m * ldy + n] += part[m * N + n];
  }
  free(part);
  if (b)
    for (int64_t m = 0; m < M; ++m)
      for (int64_t n = 0; n < N; ++n) Y[m * ldy + n] += (double)b[n];
  return ORC_OK;
}

/* Round an fp64 value to the nearest fp32 value (ties to even). */
double orc_round_f32(double x) { return (double)(float)x; }

/*
 * Row-parallel linear whose all-reduce adds the partials the way a ring
 * all-reduce does on real devices [P3 RowParallelLinear (dist.all_reduce SUM
 * of each rank's local partial, then + bias); P5 "Communication cost" (the
 * ring all-reduce: the message is cut into p chunks, each chunk's running sum
 * travels once around the ring in the reduce-scatter, the all-gather copies
 * the finished chunks)].
 *
 * Readings where the pages leave the arithmetic open:
 *   - each rank holds its partial Y_i = X_i . W_i^T in the wire dtype (fp32,
 *     or bf16 rounded to nearest even) before the collective;
 *   - every hop sends the running sum in the wire dtype, so the sum is rounded
 *     to the wire dtype after each addition;
 *   - the flattened message of L = M*N elements is cut into p chunks, chunk c
 *     = elements [c*L/p, (c+1)*L/p) (integer division);
 *   - chunk c's running sum starts with rank c's partial and adds ranks c+1,
 *     c+2, ..., c+p-1 (mod p), one per hop;
 *   - the bias is added once, after the all-reduce; this oracle returns that
 *     sum unrounded (fp64).
 * wire_bf16 != 0 selects the bf16 wire, else fp32.
 */
int orc_row_parallel_ring(int tp, int64_t M, int64_t K, int64_t N, const float* X,
                          int64_t ldx, const float* W, int64_t ldw, const float* b,
                          int wire_bf16, double* Y, int64_t ldy) {
  if (tp < 1) return ORC_ERR_BAD_SHAPE;
  if (M < 0 || K < 0 || N < 0) return ORC_ERR_BAD_SHAPE;
  if (K % tp != 0) return ORC_ERR_NOT_DIVISIBLE;
  const int64_t ks = K / tp;
  const int64_t L = M * N;
  double* part = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L * tp : 1));
  if (!part) return ORC_ERR_NOMEM;
  for (int i = 0; i < tp; ++i) {
    /* rank i's local partial, held in the wire dtype */
    double* pi = part + (int64_t)i * L;
    int rc = orc_linear(M, ks, N, X + (int64_t)i * ks, ldx, W + (int64_t)i * ks, ldw, NULL,
                        ORC_ACT_NONE, pi, N);
    if (rc != ORC_OK) {
      free(part);
      return rc;
    }
    for (int64_t e = 0; e < L; ++e) pi[e] = wire_bf16 ? orc_round_bf16(pi[e]) : orc_round_f32(pi[e]);
  }
  for (int c = 0; c < tp; ++c) {
    const int64_t e0 = (int64_t)c * L / tp, e1 = (int64_t)(c + 1) * L / tp;
    for (int64_t e = e0; e < e1; ++e) {
      double acc = part[(int64_t)c * L + e];
      for (int s = 1; s < tp; ++s) {
        const int r = (c + s) % tp;
        acc += part[(int64_t)r * L + e];
        acc = wire_bf16 ? orc_round_bf16(acc) : orc_round_f32(acc);
      }
      const int64_t m = e / N, n = e % N;
      Y[m * ldy + n] = acc + (b ? (double)b[n] : 0.0);
    }
  }
  free(part);
  return ORC_OK;
}

/*
 * The same ring-ordered all-reduce, evaluated only on some rows of a call of
 * M_total rows: X holds the n_rows sampled input rows, rows[r] is the row
 * number of sampled row r in the full call, and Y receives those output
 * rows.  The chunks are those of the full call's flattened [M_total, N]
 * message, so element (rows[r], n) is summed exactly as orc_row_parallel_ring
 * sums it in the full call; each element is computed on its own (its
 * partials, its chunk's start rank, the hops in ring order).
 */
int orc_row_parallel_ring_rows(int tp, int64_t M_total, const int64_t* rows, int64_t n_rows,
                               int64_t K, int64_t N, const float* X, int64_t ldx,
                               const float* W, int64_t ldw, const float* b, int wire_bf16,
                               double* Y, int64_t ldy) {
  if (tp < 1 || tp > 64) return ORC_ERR_BAD_SHAPE;
  if (M_total < 0 || n_rows < 0 || K < 0 || N < 0) return ORC_ERR_BAD_SHAPE;
  if (K % tp != 0) return ORC_ERR_NOT_DIVISIBLE;
  if (n_rows > 0 && !rows) return ORC_ERR_NULL;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= M_total) return ORC_ERR_BAD_SHAPE;
  const int64_t ks = K / tp;
  const int64_t L = M_total * N;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t r = 0; r < n_rows; ++r)
    for (int64_t n = 0; n < N; ++n) {
      double p[64];
      /* rank i's partial for this element, held in the wire dtype */
      for (int i = 0; i < tp; ++i) {
        const double v = dot(ks, X + r * ldx + (int64_t)i * ks, W + n * ldw + (int64_t)i * ks);
        p[i] = wire_bf16 ? orc_round_bf16(v) : orc_round_f32(v);
      }
      /* the chunk holding flattened element e of the full message */
      const int64_t e = rows[r] * N + n;
      int c = 0;
      while (c + 1 < tp && (int64_t)(c + 1) * L / tp <= e) ++c;
      double acc = p[c];
      for (int s = 1; s < tp; ++s) {
        acc += p[(c + s) % tp];
        acc = wire_bf16 ? orc_round_bf16(acc) : orc_round_f32(acc);
      }
      Y[r * ldy + n] = acc + (b ? (double)b[n] : 0.0);
    }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* FP8 (e4m3) weights with one fp32 scale per weight row                     */
/* ------------------------------------------------------------------------ */
/*
 * "Model Parallelism" (statistical-learning-notes) sizes weights at about one
 * byte per parameter in FP8; no page fixes the format or the scaling.
 * Readings: e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, largest finite value 448); one fp32 scale per weight row,
 * s = max_k |W[r,k]| / 448 (1 for an all-zero row); the code is W[r,k] / s
 * rounded to e4m3, ties to even, saturating at +-448.  The scale and the
 * division are done in fp32: that is the precision in which the code is
 * decided.  The dequantized weight is s * q.
 */

/* Round to the nearest e4m3 value, ties to even, saturating at +-448. */
double orc_round_e4m3(double x) {
  if (isnan(x) || x == 0.0) return x;
  double a = fabs(x);
  double r;
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: quantum 2^-9 */
    r = ldexp(nearbyint(ldexp(a, 9)), -9);
  } else {
    int e;
    double m = frexp(a, &e);                     /* a = m * 2^e, m in [0.5, 1) */
    r = ldexp(nearbyint(ldexp(m, 4)), e - 4);    /* keep 4 significant bits */
  }
  if (r > 448.0) r = 448.0;
  return x < 0 ? -r : r;
}

/*
 * Per-row quantization of W [rows, cols] (row stride ldw): S[r] = the row's
 * scale, Q[r*cols + c] = the e4m3 value of W[r,c] / S[r] (as a float).
 */
int orc_quantize_fp8_rows(int64_t rows, int64_t cols, const float* W, int64_t ldw, float* Q,
                          float* S) {
  if (rows < 0 || cols < 0) return ORC_ERR_BAD_SHAPE;
  if (rows * cols > 0 && (!W || !Q || !S)) return ORC_ERR_NULL;
  /* rows are independent: one row per iteration, any thread */
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    float amax = 0.0f;
    for (int64_t c = 0; c < cols; ++c) {
      const float v = fabsf(W[r * ldw + c]);
      if (v > amax) amax = v;
    }
    const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
    S[r] = sc;
    for (int64_t c = 0; c < cols; ++c) {
      const float v = W[r * ldw + c] / sc; /* fp32 division */
      Q[r * cols + c] = (float)orc_round_e4m3((double)v);
    }
  }
  return ORC_OK;
}

/*
 * Column-parallel linear with FP8 weights [the column split of
 * orc_column_parallel]: output n of shard i is act(S[n] * (x . Q[n]) + b[n]),
 * SwiGLU: silu(S[n] * (x . Q[n])) * (Su[n] * (x . Qu[n])).  Q/Qu hold the e4m3
 * values (as floats) of the unsharded [N, K] weights, S/Su their row scales;
 * shard i is rows [i*N/p, (i+1)*N/p) of each.
 */
int orc_column_parallel_fp8(int tp, int64_t M, int64_t K, int64_t N, const float* X,
                            int64_t ldx, const float* Q, const float* Qu, int64_t ldq,
                            const float* S, const float* Su, const float* b, int act, double* Y,
                            int64_t ldy) {
  if (tp < 1) return ORC_ERR_BAD_SHAPE;
  if (N % tp != 0) return ORC_ERR_NOT_DIVISIBLE;
  if (act == ORC_ACT_SWIGLU && (!Qu || !Su)) return ORC_ERR_NULL;
  const int64_t ns = N / tp;
  for (int i = 0; i < tp; ++i) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
      for (int64_t j = 0; j < ns; ++j) {
        const int64_t n = (int64_t)i * ns + j; /* row of shard i, column block i of Y */
        double z = (double)S[n] * dot(K, X + m * ldx, Q + n * ldq);
        if (act == ORC_ACT_SWIGLU) {
          const double u = (double)Su[n] * dot(K, X + m * ldx, Qu + n * ldq);
          z = orc_silu(z) * u;
        } else {
          if (b) z += (double)b[n];
          z = apply_act(act, z);
        }
        Y[m * ldy + n] = z;
      }
  }
  return ORC_OK;
}

/*
 * Row-parallel linear with FP8 weights [the row split of orc_row_parallel]:
 * shard i holds columns [i*K/p, (i+1)*K/p) of Q (e4m3 values of the
 * unsharded [N, K] weight, row stride ldq), quantized as its own [N, K/p]
 * matrix with row scales S[i*N + n].  Its partial is S_i[n] * (x_i . Q_i[n]);
 * the partials are summed in shard order, then the bias is added once.
 */
int orc_row_parallel_fp8(int tp, int64_t M, int64_t K, int64_t N, const float* X, int64_t ldx,
                         const float* Q, int64_t ldq, const float* S, const float* b, double* Y,
                         int64_t ldy) {
  if (tp < 1) return ORC_ERR_BAD_SHAPE;
  if (M < 0 || K < 0 || N < 0) return ORC_ERR_BAD_SHAPE;
  if (K % tp != 0) return ORC_ERR_NOT_DIVISIBLE;
  const int64_t ks = K / tp;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double y = 0.0;
      for (int i = 0; i < tp; ++i)
        y += (double)S[(int64_t)i * N + n] *
             dot(ks, X + m * ldx + (int64_t)i * ks, Q + n * ldq + (int64_t)i * ks);
      if (b) y += (double)b[n];
      Y[m * ldy + n] = y;
    }
  return ORC_OK;
}

/*
 * FFN block: column-parallel first linear with the nonlinearity applied per
 * shard, then row-parallel second linear whose shard-i input is h_i
 * [P3 "How Tensor Parallelism Works Under the Hood" (the FFN pairing) and its
 * demo h = gelu(ffn_up(x)); y = ffn_down(h)].
 *
 * X [M, d_model]; W1 [d_ff, d_model] (the gate weight for SwiGLU); W1u the
 * up weight for SwiGLU, else NULL; b1 [d_ff] or NULL (ignored for SwiGLU);
 * W2 [d_model, d_ff]; b2 [d_model] or NULL.
 * round_h != 0 rounds h to bf16 where the method stores it in bf16.
 * h_out (optional, [M, d_ff]) receives h after that rounding.
 */
int orc_mlp_block(int tp, int64_t M, int64_t d_model, int64_t d_ff, int act,
                  const float* X, const float* W1, const float* W1u,
                  const float* b1, const float* W2, const float* b2,
                  int round_h, double* h_out, double* Y) {
  if (tp < 1) return ORC_ERR_BAD_SHAPE;
  if (d_ff % tp != 0) return ORC_ERR_NOT_DIVISIBLE;
  if (act == ORC_ACT_SWIGLU && !W1u) return ORC_ERR_NULL;
  size_t nh = (size_t)(M * d_ff > 0 ? M * d_ff : 1);
  double* h = (double*)malloc(sizeof(double) * nh);
  float* hf = (float*)malloc(sizeof(float) * nh);
  if (!h || !hf) {
    free(h);
    free(hf);
    return ORC_ERR_NOMEM;
  }
  int rc = orc_column_parallel(tp, M, d_model, d_ff, X, d_model, W1, W1u,
                               d_model, act == ORC_ACT_SWIGLU ? NULL : b1, act,
                               h, d_ff);
  if (rc == ORC_OK) {
    for (int64_t j = 0; j < M * d_ff; ++j) {
      if (round_h) h[j] = orc_round_bf16(h[j]);
      if (h_out) h_out[j] = h[j];
    }
    /* The row layer takes float inputs.  With round_h the bf16 values are
     * exact in float.  Without it the second layer runs on the fp64 h
     * directly, so no precision is lost there either. */
    if (round_h) {
      for (int64_t j = 0; j < M * d_ff; ++j) hf[j] = (float)h[j];
      rc = orc_row_parallel(tp, M, d_ff, d_model, hf, d_ff, W2, d_ff, b2, Y,
                            d_model);
    } else {
      /* same literal split, fp64 input: partials in shard order, bias once */
      int64_t ks = d_ff / tp;
      for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < d_model; ++n) Y[m * d_model + n] = 0.0;
      for (int i = 0; i < tp; ++i) {
#pragma omp parallel for collapse(2) schedule(static)
        for (int64_t m = 0; m < M; ++m)
          for (int64_t n = 0; n < d_model; ++n) {
            double s = 0.0;
            const double* hi = h + m * d_ff + (int64_t)i * ks;
            const float* wi = W2 + n * d_ff + (int64_t)i * ks;
            for (int64_t k = 0; k < ks; ++k) s += hi[k] * (double)wi[k];
            Y[m * d_model + n] += s;
          }
      }
      if (b2)
        for (int64_t m = 0; m < M; ++m)
          for (int64_t n = 0; n < d_model; ++n) Y[m * d_model + n] += (double)b2[n];
    }
  }
  free(h);
  free(hf);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Head-split attention projections                                          */
/* ------------------------------------------------------------------------ */

/*
 * QKV projection, column-parallel by head group [P4 "How a layer is split":
 * different attention heads go to different GPUs; P4 "Why it helps when
 * serving": tp must divide the head count].
 *
 * Wqkv [(H + 2*Hkv)*hd, d_model] stores rows [Q heads; K heads; V heads].
 * Shard i gathers Q heads [i*H/p, (i+1)*H/p), then K heads and V heads
 * [i*Hkv/p, (i+1)*Hkv/p), and computes qkv_i = X . Wqkv_i^T (+ bqkv_i).
 * qkv_out is [p][M][(H + 2*Hkv)/p * hd], shard-major (what device i holds).
 */
int orc_qkv_proj(int tp, int64_t M, int64_t d_model, int H, int Hkv, int hd,
                 const float* X, const float* Wqkv, const float* bqkv,
                 double* qkv_out) {
  if (tp < 1 || H < 1 || Hkv < 1 || hd < 1) return ORC_ERR_BAD_SHAPE;
  if (H % tp != 0 || Hkv % tp != 0) return ORC_ERR_NOT_DIVISIBLE;
  int hq = H / tp, hk = Hkv / tp;
  int64_t ws = (int64_t)(hq + 2 * hk) * hd; /* rows per shard */
  for (int i = 0; i < tp; ++i) {
    double* out = qkv_out + (int64_t)i * M * ws;
    /* the three row groups of shard i, in the shard's own order Q, K, V */
    int64_t src_row[3] = {(int64_t)i * hq * hd,
                          (int64_t)H * hd + (int64_t)i * hk * hd,
                          (int64_t)(H + Hkv) * hd + (int64_t)i * hk * hd};
    int64_t nrows[3] = {(int64_t)hq * hd, (int64_t)hk * hd, (int64_t)hk * hd};
    int64_t col = 0;
    for (int g = 0; g < 3; ++g) {
      int rc = orc_linear(M, d_model, nrows[g], X, d_model,
                          Wqkv + src_row[g] * d_model, d_model,
                          bqkv ? bqkv + src_row[g] : NULL, ORC_ACT_NONE,
                          out + col, ws);
      if (rc != ORC_OK) return rc;
      col += nrows[g];
    }
  }
  return ORC_OK;
}

/*
 * Output projection, row-parallel by head [P3 "What Is Tensor Parallelism?"
 * (one exchange after the attention concatenation); P5 "Column-parallel and
 * row-parallel layers, paired" (one all-reduce per attention block)].
 * ctx [M, H*hd]; shard i owns heads [i*H/p, (i+1)*H/p), i.e. ctx columns and
 * Wo input columns [i*H/p*hd, (i+1)*H/p*hd).  Y = sum_i ctx_i . Wo_i^T + bo.
 */
int orc_o_proj(int tp, int64_t M, int64_t d_model, int H, int hd,
               const float* ctx, const float* Wo, const float* bo, double* Y) {
  if (tp < 1 || H < 1 || hd < 1) return ORC_ERR_BAD_SHAPE;
  if (H % tp != 0) return ORC_ERR_NOT_DIVISIBLE;
  int64_t K = (int64_t)H * hd;
  return orc_row_parallel(tp, M, K, d_model, ctx, K, Wo, K, bo, Y, d_model);
}
