/*
 * qlin oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU restatement of what the 8-bit quantized
 * linear layer computes.  Only the test suite, the smoke check and the timed CPU
 * baseline of the benchmark may load this file.  It shares no code, header,
 * table or constant with the CUDA library and includes no CUDA header.
 *
 * Sources (page titles as printed):
 *   [P1] "Nano-vLLM-MoE" README (English), sections "FP8 W8A16 weight-only
 *        quantization" (Setup: Triton FP8->BF16 dequant GEMM, bf16 x bf16 with
 *        fp32 accumulation) and "FP8 W8A8 static quantization" (Setup: export
 *        with offline-calibrated activation scales; _scaled_mm / CUTLASS linear
 *        backends with a custom epilogue).
 *   [P2] "Nano-vLLM-MOE" README (Chinese), section "INT8 量化支持", table
 *        "量化方案" (int8_w8a16 / int8_w8a8_static) and list "关键设计":
 *        W8A16 stores INT8 weights and dequantizes to BF16 for a standard
 *        matmul; W8A8 static calibrates one input_scale per layer offline and
 *        quantizes activations at run time with that fixed scalar, then runs
 *        an INT8 GEMM (torch._int_mm).  Calibration size from "快速使用"
 *        (--calib-samples 64 --calib-seqlen 512).
 *   The scale granularity (one scale per output channel), the formulas
 *   scale = max|row|/127 (INT8) and /448 (E4M3), symmetric clamp to
 *   [-127,127] and the saturating E4M3 cast are the method's stated
 *   definition of this layer; the pages themselves only name the schemes.
 *   E4M3 is the OCP 8-bit floating point format "E4M3" (bias 7, 3 mantissa
 *   bits, no infinities, S.1111.111 is NaN, largest finite 448, subnormal
 *   step 2^-9).
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *   - rounding of x/s to an integer is IEEE round-half-to-even (rintf);
 *   - x/s is one IEEE single-precision division (not a reciprocal multiply);
 *   - an all-zero row (or calibration batch) gets scale 1.0, so q = 0;
 *   - the E4M3 cast rounds half-to-even on the E4M3 grid, saturates
 *     magnitudes beyond 448 to 448 and keeps the sign of zero;
 *   - W8A16 applies the per-channel scale to the exact k-sum (the scale is a
 *     per-row constant, so it factors out of the sum); no intermediate BF16
 *     rounding of s*q;
 *   - the references below are computed in fp64 (exact for the integer and
 *     FP8 sums), bias added in fp64; the BF16 cast of the output is left to
 *     the comparison.
 *
 * Every function here has a pin in the not-gpu tests (brute force, closed
 * forms, invariants, an independent library cast); none is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#define ORC_INT8 0
#define ORC_E4M3 1

/* ---- BF16 storage: the upper 16 bits of an IEEE binary32 ---------------- */
static float bf16_to_f32(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* ---- OCP E4M3 ------------------------------------------------------------ */
/* Exact value of an E4M3 code (NaN for S.1111.111).  Normal: 2^(e-7)*(1+m/8)
 * = (8+m)*2^(e-10); subnormal (e=0): 2^-6*(m/8) = m*2^-9. */
double orc_e4m3_decode(uint8_t c) {
  int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
  return s ? -v : v;
}

/* Nearest E4M3 code to v, ties to the even mantissa, saturating at +-448,
 * sign of zero kept.  v is finite (NaN/Inf inputs are outside the contract). */
uint8_t orc_e4m3_encode(double v) {
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs(v);
  if (a >= 448.0) return sign | 0x7E;
  /* binade exponent E = floor(log2 a), held at the subnormal floor -6 */
  int E = -6;
  if (a > 0.0) {
    int e2;
    frexp(a, &e2); /* a = f*2^e2, f in [0.5,1) */
    if (e2 - 1 > E) E = e2 - 1;
  }
  double quantum = ldexp(1.0, E - 3); /* spacing of the grid in this binade */
  double r = nearbyint(a / quantum);  /* exact quotient; ties to even integer */
  double val = r * quantum;           /* r even <=> mantissa field even */
  if (val == 0.0) return sign;
  int e2;
  frexp(val, &e2);
  int Ev = e2 - 1;
  if (Ev < -6) return sign | (uint8_t)(val / ldexp(1.0, -9));
  int mfield = (int)(val / ldexp(1.0, Ev - 3)) - 8;
  return sign | (uint8_t)(((Ev + 7) << 3) | mfield);
}

/* ---- one quantization step: q = Q(v), v = fl32(x / s) -------------------- */
static uint8_t quantize_value(int qtype, float x, float s) {
  float v = x / s; /* one IEEE binary32 division */
  if (qtype == ORC_INT8) {
    float r = rintf(v); /* round half to even */
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    return (uint8_t)(int8_t)(int)r;
  }
  return orc_e4m3_encode((double)v);
}

static float qmax_of(int qtype) { return qtype == ORC_INT8 ? 127.0f : 448.0f; }

/* Per-output-channel symmetric weight quantization of W [N,K] (row-major fp32):
 * s[n] = fl32(max_k |w[n,k]| / QMAX); q[n,k] = Q(fl32(w[n,k] / s[n])). */
void orc_quantize_weight(int qtype, int64_t N, int64_t K, const float *w,
                         uint8_t *q, float *s) {
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) {
    const float *row = w + n * K;
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      float a = fabsf(row[k]);
      if (a > amax) amax = a;
    }
    float sn = (amax > 0.0f) ? amax / qmax_of(qtype) : 1.0f;
    s[n] = sn;
    for (int64_t k = 0; k < K; ++k) q[n * K + k] = quantize_value(qtype, row[k], sn);
  }
}

/* Static activation scale from a calibration batch x_cal [rows,K] (BF16):
 * s_x = fl32(max |x_cal| / QMAX), plain abs-max over the whole batch. */
float orc_act_scale(int qtype, int64_t rows, int64_t K, const uint16_t *x_cal) {
  float amax = 0.0f;
#pragma omp parallel for reduction(max : amax) schedule(static)
  for (int64_t i = 0; i < rows * K; ++i) {
    float a = fabsf(bf16_to_f32(x_cal[i]));
    if (a > amax) amax = a;
  }
  return (amax > 0.0f) ? amax / qmax_of(qtype) : 1.0f;
}

/* Static per-tensor activation quantization: q[m,k] = Q(fl32(x[m,k] / s_x)). */
void orc_quantize_act(int qtype, int64_t M, int64_t K, const uint16_t *x, float s_x,
                      uint8_t *q) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < M * K; ++i) q[i] = quantize_value(qtype, bf16_to_f32(x[i]), s_x);
}

/* Exact INT8 GEMM accumulator acc[m,n] = sum_k qx[m,k]*qw[n,k] (int64 sum).
 * Returns the number of entries that do not fit in int32 (0 for valid inputs:
 * |acc| <= 127*127*K < 2^31 for K < 133144). */
int64_t orc_i8_gemm(int64_t M, int64_t K, int64_t N, const int8_t *qx, const int8_t *qw,
                    int32_t *acc) {
  int64_t bad = 0;
#pragma omp parallel for reduction(+ : bad) schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      int64_t a = 0;
      for (int64_t k = 0; k < K; ++k) a += (int64_t)qx[m * K + k] * (int64_t)qw[n * K + k];
      if (a > INT32_MAX || a < INT32_MIN) ++bad;
      acc[m * N + n] = (int32_t)a;
    }
  return bad;
}

static double dequant_code(int qtype, uint8_t c) {
  return qtype == ORC_INT8 ? (double)(int8_t)c : orc_e4m3_decode(c);
}

/* Row selection: rows==NULL means all M rows, else y holds nrows output rows. */
static int64_t pick_row(const int64_t *rows, int64_t i) { return rows ? rows[i] : i; }

/* W8A8 static reference (fp64):
 *   acc = sum_k deq(qx[m,k]) * deq(qw[n,k])   (exact: int64 for INT8; for E4M3
 *         every product has <= 8 significant bits inside [2^-18, 2^17.6] and
 *         the running sum of K < 2^15 of them fits in 53 bits)
 *   y[m,n] = acc * s_x * s_w[n] + bias[n]. */
void orc_w8a8(int qtype, int64_t M, int64_t K, int64_t N, const uint8_t *qx, float s_x,
              const uint8_t *qw, const float *s_w, const uint16_t *bias,
              const int64_t *rows, int64_t nrows, double *y) {
  int64_t R = rows ? nrows : M;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t i = 0; i < R; ++i)
    for (int64_t n = 0; n < N; ++n) {
      int64_t m = pick_row(rows, i);
      double acc;
      if (qtype == ORC_INT8) {
        int64_t a = 0;
        for (int64_t k = 0; k < K; ++k)
          a += (int64_t)(int8_t)qx[m * K + k] * (int64_t)(int8_t)qw[n * K + k];
        acc = (double)a;
      } else {
        acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
          acc += orc_e4m3_decode(qx[m * K + k]) * orc_e4m3_decode(qw[n * K + k]);
      }
      double v = acc * (double)s_x * (double)s_w[n];
      if (bias) v += (double)bf16_to_f32(bias[n]);
      y[i * N + n] = v;
    }
}

/* W8A16 reference (fp64): y[m,n] = s_w[n] * sum_k x[m,k] * deq(q[n,k]) + bias[n],
 * x in BF16, q the stored 8-bit weight codes. */
void orc_w8a16(int qtype, int64_t M, int64_t K, int64_t N, const uint16_t *x,
               const uint8_t *qw, const float *s_w, const uint16_t *bias,
               const int64_t *rows, int64_t nrows, double *y) {
  int64_t R = rows ? nrows : M;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t i = 0; i < R; ++i)
    for (int64_t n = 0; n < N; ++n) {
      int64_t m = pick_row(rows, i);
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += (double)bf16_to_f32(x[m * K + k]) * dequant_code(qtype, qw[n * K + k]);
      double v = acc * (double)s_w[n];
      if (bias) v += (double)bf16_to_f32(bias[n]);
      y[i * N + n] = v;
    }
}

/* ---- dynamic per-token activation quantization -------------------------
 * The contrast the "Nano-vLLM-MOE" README draws for W8A8 static ("INT8 量化支持",
 * 关键设计, W8A8 static item): a dynamic per-token abs-max costs one more
 * reduction than the static scalar.  Per token row m:
 *   s_x[m] = fl32(max_k |x[m,k]| / QMAX)   (1 for an all-zero row)
 *   q[m,k] = Q(fl32(x[m,k] / s_x[m])). */
void orc_quantize_act_per_token(int qtype, int64_t M, int64_t K, const uint16_t *x, float *s_x,
                                uint8_t *q) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      float a = fabsf(bf16_to_f32(x[m * K + k]));
      if (a > amax) amax = a;
    }
    const float s = (amax > 0.0f) ? amax / qmax_of(qtype) : 1.0f;
    s_x[m] = s;
    for (int64_t k = 0; k < K; ++k) q[m * K + k] = quantize_value(qtype, bf16_to_f32(x[m * K + k]), s);
  }
}

/* W8A8 with one activation scale per token row:
 *   y[m,n] = acc[m,n] * s_x[m] * s_w[n] + bias[n]   (acc as in orc_w8a8). */
void orc_w8a8_per_token(int qtype, int64_t M, int64_t K, int64_t N, const uint8_t *qx, const float *s_x,
                        const uint8_t *qw, const float *s_w, const uint16_t *bias, const int64_t *rows,
                        int64_t nrows, double *y) {
  int64_t R = rows ? nrows : M;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t i = 0; i < R; ++i)
    for (int64_t n = 0; n < N; ++n) {
      int64_t m = pick_row(rows, i);
      double acc;
      if (qtype == ORC_INT8) {
        int64_t a = 0;
        for (int64_t k = 0; k < K; ++k)
          a += (int64_t)(int8_t)qx[m * K + k] * (int64_t)(int8_t)qw[n * K + k];
        acc = (double)a;
      } else {
        acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
          acc += orc_e4m3_decode(qx[m * K + k]) * orc_e4m3_decode(qw[n * K + k]);
      }
      double v = acc * (double)s_x[m] * (double)s_w[n];
      if (bias) v += (double)bf16_to_f32(bias[n]);
      y[i * N + n] = v;
    }
}

/* ---- merged gate_up linear with the SiLU * up epilogue -------------------
 * The "tiny-vLLM" README's quality check quantizes 112 target layers of the
 * 28-layer model, four linears per layer: merged qkv, o, merged gate_up, down.
 * The MLP of that model family is down(silu(gate(x)) * up(x)) with the merged
 * weight qw [2I, K] holding the gate rows [0, I) above the up rows [I, 2I).
 * Reading: the fused epilogue applies the activation to the linear's exact
 * outputs (no BF16 rounding of gate or up in between):
 *   y[m, n] = silu(g) * u,  g = lin[m, n],  u = lin[m, I + n],
 *   silu(g) = g / (1 + exp(-g)),  all in fp64;
 * lin is the W8A16 or W8A8 reference above over N = 2I channels, with the
 * optional bias [2I] added before the activation. */
static double silu(double g) { return g / (1.0 + exp(-g)); }

static void glu_combine(int64_t R, int64_t I, const double *lin, double *y) {
  for (int64_t i = 0; i < R; ++i)
    for (int64_t n = 0; n < I; ++n) y[i * I + n] = silu(lin[i * 2 * I + n]) * lin[i * 2 * I + I + n];
}

/* Returns 0 on success, -1 if the temporary [rows, 2I] buffer cannot be allocated. */
int orc_w8a16_gate_up_silu(int qtype, int64_t M, int64_t K, int64_t I, const uint16_t *x, const uint8_t *qw,
                           const float *s_w, const uint16_t *bias, const int64_t *rows, int64_t nrows, double *y) {
  int64_t R = rows ? nrows : M;
  double *lin = (double *)malloc((size_t)(R > 0 ? R : 1) * (size_t)(2 * I) * sizeof(double));
  if (!lin) return -1;
  orc_w8a16(qtype, M, K, 2 * I, x, qw, s_w, bias, rows, nrows, lin);
  glu_combine(R, I, lin, y);
  free(lin);
  return 0;
}

int orc_w8a8_gate_up_silu(int qtype, int64_t M, int64_t K, int64_t I, const uint8_t *qx, float s_x,
                          const uint8_t *qw, const float *s_w, const uint16_t *bias, const int64_t *rows,
                          int64_t nrows, double *y) {
  int64_t R = rows ? nrows : M;
  double *lin = (double *)malloc((size_t)(R > 0 ? R : 1) * (size_t)(2 * I) * sizeof(double));
  if (!lin) return -1;
  orc_w8a8(qtype, M, K, 2 * I, qx, s_x, qw, s_w, bias, rows, nrows, lin);
  glu_combine(R, I, lin, y);
  free(lin);
  return 0;
}

/* Threads the OpenMP runtime will use (1 when built without OpenMP). */
int orc_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---- mixed KV-cache quantization -----------------------------------------
 * "Nano-vLLM-MoE" README (English), section "KV cache compression" (Setup and
 * the memory table) and the Highlights list: keys are stored as INT8 with one
 * float16 scale per group of 32 consecutive head_dim elements, values as FP8
 * (E4M3) with one dynamic float16 scale per token and kv head.  This layout is
 * the one whose size matches the printed 0.5195x BF16 bytes per block and the
 * 7.00 -> 3.64 GiB arena of a 7B model (4 kv heads, head_dim 128).
 * Readings where the page is silent:
 *   - scale = RN_fp16(fl32(amax / QMAX)): an fp32 division, then the float16
 *     cast of that quotient; magnitudes beyond 65504 saturate to 65504;
 *   - a scale that is zero after the cast (all-zero group, or amax so small
 *     that amax/QMAX underflows float16) is replaced by 1.0, so the codes are 0;
 *   - codes quantize with the stored float16 scale: q = Q(fl32(x / s16));
 *   - dequantized values are the exact product q * s16 rounded once to BF16. */

/* Nearest value to a >= 0 on a binary grid with P significant bits whose
 * smallest normal exponent is EMIN (subnormals below it), ties to the even
 * last bit.  The grid spacing in the binade [2^E, 2^(E+1)) is 2^(E-P+1). */
static double round_to_grid(double a, int P, int EMIN) {
  if (a == 0.0) return 0.0;
  int e2;
  frexp(a, &e2);
  int E = e2 - 1;
  if (E < EMIN) E = EMIN;
  double quantum = ldexp(1.0, E - P + 1);
  return nearbyint(a / quantum) * quantum; /* a/quantum is exact (power of two) */
}

/* IEEE binary16: bias 15, 10 stored mantissa bits, subnormal step 2^-24,
 * largest finite 65504.  Exact value of a finite code (NaN/Inf map to NaN/Inf). */
double orc_fp16_decode(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 31) v = m ? NAN : INFINITY;
  else v = (e == 0) ? ldexp((double)m, -24) : ldexp((double)(1024 + m), e - 25);
  return s ? -v : v;
}

/* Nearest binary16 code to a finite v, ties to even, saturating at +-65504,
 * sign of zero kept. */
uint16_t orc_fp16_encode(double v) {
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = round_to_grid(fabs(v), 11, -14);
  if (a >= 65504.0) return sign | 0x7BFF;
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);
  int E = e2 - 1;
  if (E < -14) return sign | (uint16_t)(a / ldexp(1.0, -24)); /* subnormal */
  int mfield = (int)(a / ldexp(1.0, E - 10)) - 1024;
  return sign | (uint16_t)(((E + 15) << 10) | mfield);
}

/* BF16 (the upper half of binary32: 8 significant bits, exponent range of
 * fp32) nearest to a finite v inside the binary32 range, ties to even. */
uint16_t orc_bf16_encode(double v) {
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = round_to_grid(fabs(v), 8, -126);
  float f = (float)a; /* exact: a lies on the BF16 grid */
  uint32_t u;
  memcpy(&u, &f, 4);
  return sign | (uint16_t)(u >> 16);
}

static uint16_t kv_scale16(float amax, float qmax) {
  float s32 = amax / qmax; /* IEEE binary32 division */
  uint16_t h = orc_fp16_encode((double)s32);
  if ((h & 0x7FFF) == 0) h = 0x3C00; /* 1.0 */
  return h;
}

/* Quantizes the T token rows of k and v (BF16, row t at k + t*ldk, holding H
 * heads of D elements each; D a multiple of 32) into the slots slots[t] of a
 * cache with num_slots slots:
 *   k_cache[slot][h][d] int8, k_scale[slot][h][d/32] float16 bits,
 *   v_cache[slot][h][d] E4M3, v_scale[slot][h] float16 bits.
 * A negative slot skips the token.  Returns the number of tokens whose slot is
 * >= num_slots (those are skipped too). */
int64_t orc_kv_store(int64_t T, int64_t H, int64_t D, const uint16_t *k, int64_t ldk,
                     const uint16_t *v, int64_t ldv, const int64_t *slots, int64_t num_slots,
                     uint8_t *k_cache, uint16_t *k_scale, uint8_t *v_cache, uint16_t *v_scale) {
  const int64_t G = D / 32;
  int64_t bad = 0;
  for (int64_t t = 0; t < T; ++t) {
    int64_t slot = slots[t];
    if (slot < 0) continue;
    if (slot >= num_slots) { ++bad; continue; }
    for (int64_t h = 0; h < H; ++h) {
      const uint16_t *kr = k + t * ldk + h * D;
      const uint16_t *vr = v + t * ldv + h * D;
      uint8_t *kq = k_cache + (slot * H + h) * D;
      uint8_t *vq = v_cache + (slot * H + h) * D;
      for (int64_t g = 0; g < G; ++g) {
        float amax = 0.0f;
        for (int64_t d = 32 * g; d < 32 * g + 32; ++d) {
          float a = fabsf(bf16_to_f32(kr[d]));
          if (a > amax) amax = a;
        }
        uint16_t s16 = kv_scale16(amax, 127.0f);
        k_scale[(slot * H + h) * G + g] = s16;
        float s = (float)orc_fp16_decode(s16);
        for (int64_t d = 32 * g; d < 32 * g + 32; ++d) kq[d] = quantize_value(ORC_INT8, bf16_to_f32(kr[d]), s);
      }
      float amax = 0.0f;
      for (int64_t d = 0; d < D; ++d) {
        float a = fabsf(bf16_to_f32(vr[d]));
        if (a > amax) amax = a;
      }
      uint16_t s16 = kv_scale16(amax, 448.0f);
      v_scale[slot * H + h] = s16;
      float s = (float)orc_fp16_decode(s16);
      for (int64_t d = 0; d < D; ++d) vq[d] = quantize_value(ORC_E4M3, bf16_to_f32(vr[d]), s);
    }
  }
  return bad;
}

/* Reads slots[t] of the cache back as BF16 rows k_out[t][h][d], v_out[t][h][d]
 * (row stride H*D): value = RN_bf16(code * scale), exact product.  A negative
 * slot yields a row of +0.  Returns the number of slots >= num_slots (their
 * rows are left as +0 too). */
int64_t orc_kv_load(int64_t T, int64_t H, int64_t D, const int64_t *slots, int64_t num_slots,
                    const uint8_t *k_cache, const uint16_t *k_scale, const uint8_t *v_cache,
                    const uint16_t *v_scale, uint16_t *k_out, uint16_t *v_out) {
  const int64_t G = D / 32;
  int64_t bad = 0;
  for (int64_t t = 0; t < T; ++t) {
    int64_t slot = slots[t];
    int ok = slot >= 0 && slot < num_slots;
    if (slot >= num_slots) ++bad;
    for (int64_t h = 0; h < H; ++h)
      for (int64_t d = 0; d < D; ++d) {
        int64_t o = (t * H + h) * D + d;
        if (!ok) { k_out[o] = 0; v_out[o] = 0; continue; }
        int64_t c = (slot * H + h) * D + d;
        double ks = orc_fp16_decode(k_scale[(slot * H + h) * G + d / 32]);
        double vs = orc_fp16_decode(v_scale[slot * H + h]);
        k_out[o] = orc_bf16_encode((double)(int8_t)k_cache[c] * ks);
        v_out[o] = orc_bf16_encode(orc_e4m3_decode(v_cache[c]) * vs);
      }
  }
  return bad;
}
