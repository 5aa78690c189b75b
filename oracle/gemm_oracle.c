/*
 * Plain CPU oracle for the tiled GEMM  D = act(alpha * A * B + beta * C + bias).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product (the CUDA
 * library and its Python binding) never calls it and shares no code with it.
 *
 * What it follows (page: "CUTLASS tutorial: from hand-written GEMM to CuTe /
 * Tensor Core kernels", hpc.payai.win/cutlass):
 *   - section 1, "map the GEMM triple loop onto the GPU hierarchy":
 *     C[M,N] = A[M,K] x B[K,N], i.e. s_ij = sum_k a_ik * b_kj;
 *   - same section, Epilogue box: alpha/beta, then bias/activation, then store;
 *   - section 2, device::Gemm: a host entry with cuBLAS-like semantics
 *     (alpha scales the product, beta scales the existing C).
 * Readings where the pages are silent:
 *   - bias is fp32[N], added per output column after alpha/beta;
 *   - the activation is ReLU = max(v, 0) or the tanh form of GELU,
 *     0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)));
 *   - beta == 0 means C is not read at all (BLAS convention);
 *   - storage: row-major element (i, j) at i*ld + j, column-major at i + j*ld.
 *
 * Arithmetic: every stored input is widened exactly to double (fp16/bf16) or
 * int64 (int8); the dot product is a plain sequential loop over k in that
 * precision; the epilogue runs in double with libm's tanh.  The returned value
 * is the UNROUNDED result r (the caller compares the GPU's rounded output to
 * it).  Alongside r the loop returns S_abs = sum_k |a_ik * b_kj|, which the
 * tolerance of the float path is stated in.
 *
 * Nothing here is blocked, fused or reordered: each requested element is one
 * independent loop.  Work is split over threads by element only.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { OR_F16 = 0, OR_BF16 = 1, OR_I8 = 2 };
enum { OR_ROW = 0, OR_COL = 1 };
enum { OR_ACT_NONE = 0, OR_ACT_RELU = 1, OR_ACT_GELU_TANH = 2 };

/* IEEE 754 binary16 -> double, from the format's definition (exact). */
double oracle_f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int f = h & 0x3FF;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(f + 1024), e - 25); /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16 -> double: bfloat16 is the upper half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t h) {
  uint32_t bits = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static int64_t offset_of(int layout, int64_t ld, int64_t i, int64_t j) {
  return layout == OR_ROW ? i * ld + j : i + j * ld;
}

static double load_float(const void* p, int dtype, int64_t idx) {
  uint16_t h = ((const uint16_t*)p)[idx];
  return dtype == OR_F16 ? oracle_f16_to_double(h) : oracle_bf16_to_double(h);
}

double oracle_gelu_tanh(double v) {
  const double k0 = sqrt(2.0 / M_PI);
  return 0.5 * v * (1.0 + tanh(k0 * (v + 0.044715 * v * v * v)));
}

double oracle_act(int act, double v) {
  if (act == OR_ACT_RELU) return v > 0.0 ? v : 0.0;
  if (act == OR_ACT_GELU_TANH) return oracle_gelu_tanh(v);
  return v;
}

typedef struct {
  int64_t M, N, K;
  const void* A; int64_t lda; int layA;
  const void* B; int64_t ldb; int layB;
  const void* C; int64_t ldc;
  float alpha, beta;
  const float* bias;
  int act, dtype;
  int64_t n;
  const int64_t* ii;
  const int64_t* jj;
  double* r;
  double* sabs;
} gemm_job;

typedef struct {
  const gemm_job* job;
  int64_t lo, hi;
} gemm_slice;

/* One output element, straight from the definition. */
static void one_element(const gemm_job* g, int64_t i, int64_t j, double* r, double* sabs) {
  double v;
  double a_abs = 0.0;
  if (g->dtype == OR_I8) {
    const int8_t* A = (const int8_t*)g->A;
    const int8_t* B = (const int8_t*)g->B;
    int64_t s = 0, sa = 0;
    for (int64_t k = 0; k < g->K; ++k) {
      int64_t p = (int64_t)A[offset_of(g->layA, g->lda, i, k)] *
                  (int64_t)B[offset_of(g->layB, g->ldb, k, j)];
      s += p;
      sa += p < 0 ? -p : p;
    }
    v = (double)g->alpha * (double)s;
    if (g->beta != 0.0f) v += (double)g->beta * (double)((const int32_t*)g->C)[i * g->ldc + j];
    a_abs = (double)sa;
  } else {
    double s = 0.0;
    for (int64_t k = 0; k < g->K; ++k) {
      double p = load_float(g->A, g->dtype, offset_of(g->layA, g->lda, i, k)) *
                 load_float(g->B, g->dtype, offset_of(g->layB, g->ldb, k, j));
      s += p;
      a_abs += fabs(p);
    }
    v = (double)g->alpha * s;
    if (g->beta != 0.0f) v += (double)g->beta * load_float(g->C, g->dtype, i * g->ldc + j);
  }
  if (g->bias) v += (double)g->bias[j];
  *r = oracle_act(g->act, v);
  *sabs = a_abs;
}

static void* run_slice(void* arg) {
  const gemm_slice* s = (const gemm_slice*)arg;
  const gemm_job* g = s->job;
  for (int64_t e = s->lo; e < s->hi; ++e) one_element(g, g->ii[e], g->jj[e], &g->r[e], &g->sabs[e]);
  return NULL;
}

int oracle_num_cpus(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/*
 * Computes r and S_abs for the n output elements (ii[e], jj[e]).
 * C is row-major with ldc and has the input dtype for fp16/bf16, int32 for
 * int8; it is read only when beta != 0.  bias may be NULL.
 * nthreads <= 0 uses every online core.  Returns the thread count used.
 */
int oracle_gemm_elements(int64_t M, int64_t N, int64_t K,
                         const void* A, int64_t lda, int layA,
                         const void* B, int64_t ldb, int layB,
                         const void* C, int64_t ldc,
                         float alpha, float beta, const float* bias,
                         int act, int dtype,
                         int64_t n, const int64_t* ii, const int64_t* jj,
                         double* r, double* sabs, int nthreads) {
  gemm_job g = {M, N, K, A, lda, layA, B, ldb, layB, C, ldc, alpha, beta, bias,
                act, dtype, n, ii, jj, r, sabs};
  if (nthreads <= 0) nthreads = oracle_num_cpus();
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > n) nthreads = n > 0 ? (int)n : 1;
  pthread_t th[256];
  gemm_slice sl[256];
  for (int t = 0; t < nthreads; ++t) {
    sl[t].job = &g;
    sl[t].lo = n * t / nthreads;
    sl[t].hi = n * (t + 1) / nthreads;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, run_slice, &sl[t]);
  run_slice(&sl[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  return nthreads;
}

/*
 * y = X x in double for a logical rows x cols matrix X stored with (layout,
 * ld) in dtype (fp16/bf16/int8 widened exactly).  Used by the Freivalds
 * check A (B x) of a full output: the definition of a matrix-vector product.
 */
void oracle_matvec(int64_t rows, int64_t cols, const void* X, int64_t ld, int layout,
                   int dtype, const double* x, double* y) {
  for (int64_t i = 0; i < rows; ++i) {
    double s = 0.0;
    for (int64_t j = 0; j < cols; ++j) {
      int64_t o = offset_of(layout, ld, i, j);
      double xv = dtype == OR_I8 ? (double)((const int8_t*)X)[o] : load_float(X, dtype, o);
      s += xv * x[j];
    }
    y[i] = s;
  }
}

/*
 * 2-D convolution, forward (cross-correlation), from its textbook definition.
 * The PitchLinearStripminedThreadMap walkthrough (lpnh.cn/news/2469163),
 * section 5.2, describes the implicit-GEMM view of it: one GEMM dimension is
 * the output pixel, the other the filter tap x channel combination, and the
 * loads follow the filter's sliding window.  The pages give no formula; this
 * is the standard one:
 *   P = (H + 2 ph - dh (R - 1) - 1) / sh + 1,  Q = (W + 2 pw - dw (S - 1) - 1) / sw + 1
 *   acc[n, p, q, k] = sum over r < R, s < S, c < C of
 *                     x[n, p sh - ph + r dh, q sw - pw + s dw, c] * w[k, r, s, c]
 * where taps that fall outside the H x W input contribute nothing (zero
 * padding).  x is NHWC and w is KRSC, both tightly packed.  The output is the
 * (N P Q) x K matrix with row m = (n P + p) Q + q, and the GEMM's epilogue
 * applies: act(alpha acc + beta C[m, k] + bias[k]) (C row-major, pitch ldc,
 * read only when beta != 0).  fp16/bf16 inputs widen exactly to double; one
 * sequential loop over (r, s, c) per element; S_abs = sum |x w| as for the GEMM.
 */
typedef struct {
  int64_t N, H, W, C, K, R, S, P, Q;
  int64_t ph, pw, sh, sw, dh, dw;
  const void* X;
  const void* Wt;
  const void* Cm;
  int64_t ldc;
  float alpha, beta;
  const float* bias;
  int act, dtype;
  int64_t n;
  const int64_t* mm;
  const int64_t* kk;
  double* r;
  double* sabs;
} conv_job;

typedef struct {
  const conv_job* job;
  int64_t lo, hi;
} conv_slice;

int64_t oracle_conv_out_extent(int64_t in, int64_t pad, int64_t dil, int64_t taps, int64_t stride) {
  int64_t span = in + 2 * pad - dil * (taps - 1) - 1;
  return span < 0 ? 0 : span / stride + 1;
}

static void conv_one(const conv_job* g, int64_t m, int64_t k, double* r, double* sabs) {
  const int64_t n = m / (g->P * g->Q);
  const int64_t p = (m / g->Q) % g->P;
  const int64_t q = m % g->Q;
  double s = 0.0, a_abs = 0.0;
  for (int64_t rr = 0; rr < g->R; ++rr) {
    const int64_t h = p * g->sh - g->ph + rr * g->dh;
    if (h < 0 || h >= g->H) continue;
    for (int64_t ss = 0; ss < g->S; ++ss) {
      const int64_t w = q * g->sw - g->pw + ss * g->dw;
      if (w < 0 || w >= g->W) continue;
      for (int64_t c = 0; c < g->C; ++c) {
        const double xv = load_float(g->X, g->dtype, ((n * g->H + h) * g->W + w) * g->C + c);
        const double wv = load_float(g->Wt, g->dtype, ((k * g->R + rr) * g->S + ss) * g->C + c);
        s += xv * wv;
        a_abs += fabs(xv * wv);
      }
    }
  }
  double v = (double)g->alpha * s;
  if (g->beta != 0.0f) v += (double)g->beta * load_float(g->Cm, g->dtype, m * g->ldc + k);
  if (g->bias) v += (double)g->bias[k];
  *r = oracle_act(g->act, v);
  *sabs = a_abs;
}

static void* conv_run_slice(void* arg) {
  const conv_slice* s = (const conv_slice*)arg;
  const conv_job* g = s->job;
  for (int64_t e = s->lo; e < s->hi; ++e) conv_one(g, g->mm[e], g->kk[e], &g->r[e], &g->sabs[e]);
  return NULL;
}

/*
 * r and S_abs for the n output elements (mm[e], kk[e]) of the convolution
 * above (fp16 or bf16 only).  Returns the thread count used, or -1 when the
 * output would be empty.
 */
int oracle_conv2d_elements(int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R, int64_t S,
                           int64_t ph, int64_t pw, int64_t sh, int64_t sw, int64_t dh, int64_t dw,
                           const void* X, const void* Wt, const void* Cm, int64_t ldc,
                           float alpha, float beta, const float* bias, int act, int dtype,
                           int64_t n, const int64_t* mm, const int64_t* kk,
                           double* r, double* sabs, int nthreads) {
  conv_job g;
  g.N = N; g.H = H; g.W = W; g.C = C; g.K = K; g.R = R; g.S = S;
  g.P = oracle_conv_out_extent(H, ph, dh, R, sh);
  g.Q = oracle_conv_out_extent(W, pw, dw, S, sw);
  if (g.P <= 0 || g.Q <= 0) return -1;
  g.ph = ph; g.pw = pw; g.sh = sh; g.sw = sw; g.dh = dh; g.dw = dw;
  g.X = X; g.Wt = Wt; g.Cm = Cm; g.ldc = ldc;
  g.alpha = alpha; g.beta = beta; g.bias = bias; g.act = act; g.dtype = dtype;
  g.n = n; g.mm = mm; g.kk = kk; g.r = r; g.sabs = sabs;
  if (nthreads <= 0) nthreads = oracle_num_cpus();
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > n) nthreads = n > 0 ? (int)n : 1;
  pthread_t th[256];
  conv_slice sl[256];
  for (int t = 0; t < nthreads; ++t) {
    sl[t].job = &g;
    sl[t].lo = n * t / nthreads;
    sl[t].hi = n * (t + 1) / nthreads;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, conv_run_slice, &sl[t]);
  conv_run_slice(&sl[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  return nthreads;
}
