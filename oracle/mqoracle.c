/*
 * mqoracle.c -- plain CPU oracle for MicroQonv quantize-once + convolution.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  It shares
 * no code, header, table or constant generator with the CUDA path.
 *
 * Everything here is written to be checked by eye against the paper
 * "MicroQonv: Reshaping Convolution Tensors for Efficient Microscaling in
 * Training and Inference" (Facq, Ben Ali, Sentieys):
 *
 *   - element formats and the two-level NVFP4-style scaling:
 *       MicroQonv §II-D (Quantization) and §III-A (Microscaling quantization):
 *       T_scale from amax / (maxB_ef * maxB_sf), maxB_sf = 448 (E4M3),
 *       maxB_ef = 6 (E2M1); B_scale = CastE4M3(amax(X_i) / (maxB_ef * T_scale));
 *       X_i^q = Round(X_i / (B_scale * T_scale)); fake quantization multiplies
 *       X_i^q back by B_scale * T_scale.
 *   - square 8x8 blocks, B = 64, and the block directions per tensor:
 *       MicroQonv §IV-B (Efficient quantization directions).
 *   - channel-batch-first storage: MicroQonv §IV-A and Fig. 3.
 *   - the three convolution GEMMs: MicroQonv §II-A, §II-C and §IV-A
 *       (Y = W * X', G_W = G_Y * X'^T, G_X' = W^T * G_Y); output size
 *       Hout = Hin - Kh + 1 at stride 1 without padding (paperlayer summary,
 *       §II-A "Forward Pass"), generalised to floor((H + 2p - K) / s) + 1 as
 *       the paper states its method is independent of stride and padding.
 *
 * Readings taken where the pages are silent:
 *   - T_scale = fl32(amax / (maxB_ef * 448)): one correctly rounded fp32 division.
 *   - Both roundings act on the exact real quotient (no intermediate rounded
 *     quotient), nearest grid value, ties to the code with an even mantissa,
 *     values past the largest finite value clamp to it (satfinite).
 *   - A block whose scale rounds to 0 (or a tensor with T_scale = 0) gets
 *     magnitude-0 codes.  The sign bit of every code is the sign bit of its input.
 *   - Element order inside a block: activations/gradients [n][c] (channel
 *     fastest), weights [c_out][c_in] (c_in fastest); block order
 *     [H][W][N/8][C/8] for activations/gradients, [Kh][Kw][Cout/8][Cin/8] for
 *     weights.  FP4 packs element i in byte i/2 (low nibble for even i); FP6
 *     is a little-endian bit stream (element i at bits 6i..6i+5); FP8 is one
 *     byte per element.  Block scales are one E4M3 byte per block, in block order.
 *
 * Why fp64 division is exact enough for the rounding decisions: the quotient
 * x / d has x with 24 significant bits and d = B_scale * T_scale (or
 * maxB_ef * T_scale) with at most 28; a rounding midpoint m of the grid has at
 * most 5.  If x / d != m then |x - m d| >= 2^-34 |x|, far larger than the
 * 2^-53 relative error of one fp64 division, so the fp64 quotient lies on the
 * same side of every midpoint as the exact one, and equals m exactly when the
 * exact quotient does.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_NONFINITE 2

/* element formats, identified by their bit width */
#define ORC_E2M1 4
#define ORC_E2M3 6
#define ORC_E4M3 8

#define ORC_ROLE_ACT 0
#define ORC_ROLE_WEIGHT 1
#define ORC_ROLE_GRAD 2

#define ORC_NCHW 0
#define ORC_HWCN 1
#define ORC_OIHW 2

/* ---------------------------------------------------------------- formats */

typedef struct {
  int ebits, mbits, bias;
  int fn_nan; /* 1: the all-ones exponent+mantissa pattern is NaN (E4M3 "FN") */
} fmt_t;

static int fmt_get(int fmt, fmt_t *f) {
  switch (fmt) {
    case ORC_E2M1: f->ebits = 2; f->mbits = 1; f->bias = 1; f->fn_nan = 0; return 1;
    case ORC_E2M3: f->ebits = 2; f->mbits = 3; f->bias = 1; f->fn_nan = 0; return 1;
    case ORC_E4M3: f->ebits = 4; f->mbits = 3; f->bias = 7; f->fn_nan = 1; return 1;
    default: return 0;
  }
}

/* value of a magnitude code (sign bit excluded): the usual minifloat rule,
 * subnormal when the exponent field is 0 */
static double fmt_mag_value(const fmt_t *f, unsigned mag) {
  unsigned e = mag >> f->mbits, m = mag & ((1u << f->mbits) - 1u);
  if (e == 0) return ldexp((double)m, 1 - f->bias - f->mbits);
  return ldexp(1.0 + ldexp((double)m, -f->mbits), (int)e - f->bias);
}

/* number of finite magnitude codes: 0 .. count-1 are finite and increasing */
static int fmt_count(const fmt_t *f) {
  int n = 1 << (f->ebits + f->mbits);
  return f->fn_nan ? n - 1 : n;
}

/* The finite non-negative grid, indexed by magnitude code. */
int orc_format_grid(int fmt, double *mags, int *count) {
  fmt_t f;
  if (!fmt_get(fmt, &f)) return ORC_ERR_ARG;
  int n = fmt_count(&f);
  for (int i = 0; i < n; ++i) mags[i] = fmt_mag_value(&f, (unsigned)i);
  *count = n;
  return ORC_OK;
}

/* Round a non-negative fp64 value to the nearest finite grid value; ties go
 * to the even magnitude code; anything above the largest value clamps to it. */
static unsigned round_mag(const double *grid, int n, double q) {
  if (!(q > 0.0)) return 0u;
  if (q >= grid[n - 1]) return (unsigned)(n - 1);
  int lo = 0, hi = n - 1; /* invariant: grid[lo] <= q < grid[hi] */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (grid[mid] <= q) lo = mid; else hi = mid;
  }
  double midpoint = 0.5 * (grid[lo] + grid[hi]); /* exact: few significant bits */
  if (q < midpoint) return (unsigned)lo;
  if (q > midpoint) return (unsigned)hi;
  return (lo & 1) ? (unsigned)hi : (unsigned)lo;
}

/* Codes (sign bit | magnitude code) for an array of fp64 values. */
int orc_round(int fmt, const double *q, int64_t n, uint8_t *codes) {
  fmt_t f;
  double grid[256];
  if (!fmt_get(fmt, &f)) return ORC_ERR_ARG;
  int cnt = fmt_count(&f);
  for (int i = 0; i < cnt; ++i) grid[i] = fmt_mag_value(&f, (unsigned)i);
  unsigned sbit = 1u << (f.ebits + f.mbits);
  for (int64_t i = 0; i < n; ++i) {
    unsigned c = round_mag(grid, cnt, fabs(q[i]));
    if (signbit(q[i])) c |= sbit;
    codes[i] = (uint8_t)c;
  }
  return ORC_OK;
}

/* Signed value of a code. */
int orc_decode(int fmt, const uint8_t *codes, int64_t n, double *out) {
  fmt_t f;
  if (!fmt_get(fmt, &f)) return ORC_ERR_ARG;
  unsigned sbit = 1u << (f.ebits + f.mbits);
  for (int64_t i = 0; i < n; ++i) {
    double v = fmt_mag_value(&f, codes[i] & (sbit - 1u));
    out[i] = (codes[i] & sbit) ? -v : v;
  }
  return ORC_OK;
}

/* largest finite element value: maxB_ef of MicroQonv §III-A */
static double fmt_max(const fmt_t *f) { return fmt_mag_value(f, (unsigned)(fmt_count(f) - 1)); }

/* T_scale = fl32(amax / (maxB_ef * maxB_sf)), maxB_sf = 448 (E4M3) */
float orc_tensor_scale(int fmt, float amax) {
  fmt_t f;
  if (!fmt_get(fmt, &f)) return -1.0f;
  float denom = (float)(fmt_max(&f) * 448.0); /* 2688, 3360 or 200704: exact */
  volatile float q = amax / denom;           /* one IEEE fp32 division */
  return q;
}

/* ------------------------------------------------------- block geometry */

static int64_t block_bytes(int fmt) { return fmt == ORC_E2M1 ? 32 : fmt == ORC_E2M3 ? 48 : 64; }

int64_t orc_num_blocks(int role, const int64_t d[4]) {
  /* ACT/GRAD: d = (N, C, H, W); WEIGHT: d = (Cout, Cin, Kh, Kw) */
  (void)role;
  return (d[0] / 8) * (d[1] / 8) * d[2] * d[3];
}

/* index of element (a, b, s0, s1) in the dense source layout.
 *   ACT/GRAD: a = n, b = c, (s0, s1) = (h, w);  layout NCHW or HWCN
 *   WEIGHT:   a = co, b = ci, (s0, s1) = (kh, kw); layout OIHW            */
static int64_t src_index(int layout, const int64_t d[4], int64_t a, int64_t b, int64_t s0, int64_t s1) {
  if (layout == ORC_HWCN) return ((s0 * d[3] + s1) * d[1] + b) * d[0] + a;
  return ((a * d[1] + b) * d[2] + s0) * d[3] + s1; /* NCHW and OIHW */
}

/* block (s0, s1, ga, gb) -> linear block index.  ACT/GRAD blocks are ordered
 * [H][W][N/8][C/8]; weight blocks [Kh][Kw][Cout/8][Cin/8].  Both are
 * [s0][s1][a/8][b/8] with a = n or co, b = c or ci. */
static int64_t block_index(const int64_t d[4], int64_t s0, int64_t s1, int64_t ga, int64_t gb) {
  return ((s0 * d[3] + s1) * (d[0] / 8) + ga) * (d[1] / 8) + gb;
}

static void put_code(int fmt, uint8_t *blk, int i, unsigned code) {
  if (fmt == ORC_E2M1) {
    blk[i / 2] |= (uint8_t)(code << (4 * (i & 1)));
  } else if (fmt == ORC_E2M3) {
    for (int j = 0; j < 6; ++j) {
      int bit = 6 * i + j;
      blk[bit / 8] |= (uint8_t)(((code >> j) & 1u) << (bit % 8));
    }
  } else {
    blk[i] = (uint8_t)code;
  }
}

static unsigned get_code(int fmt, const uint8_t *blk, int i) {
  if (fmt == ORC_E2M1) return (blk[i / 2] >> (4 * (i & 1))) & 0xFu;
  if (fmt == ORC_E2M3) {
    unsigned c = 0;
    for (int j = 0; j < 6; ++j) {
      int bit = 6 * i + j;
      c |= ((blk[bit / 8] >> (bit % 8)) & 1u) << j;
    }
    return c;
  }
  return blk[i];
}

static int valid_dims(int role, const int64_t d[4]) {
  (void)role;
  return d[0] > 0 && d[1] > 0 && d[2] > 0 && d[3] > 0 && d[0] % 8 == 0 && d[1] % 8 == 0;
}

/* ------------------------------------------------------------- quantizer */

/*
 * Quantize one tensor once into square 8x8 blocks (MicroQonv §III-A, §IV-B).
 * src: dense fp32 in `layout`.  amax_in: NULL to use the tensor's own amax,
 * else the value to build T_scale from (statistics supplied by the caller, as
 * in the Hindsight scheme the paper uses in §VII).  Writes codes, one E4M3
 * scale byte per block, T_scale, and the tensor's measured amax.
 */
static unsigned sr_round_mag(const double *grid, int n, float ax, float bs, float s_t, uint32_t word);
static uint32_t philox_word(uint64_t seed, int64_t index);

static int quantize_impl(const float *src, int layout, int role, int fmt, const int64_t d[4],
                         const float *amax_in, uint8_t *codes, uint8_t *scales,
                         float *s_t_out, float *amax_out, int stochastic, uint64_t seed) {
  fmt_t f, f8;
  if (!fmt_get(fmt, &f) || !fmt_get(ORC_E4M3, &f8) || !valid_dims(role, d)) return ORC_ERR_ARG;
  if ((role == ORC_ROLE_WEIGHT) != (layout == ORC_OIHW)) return ORC_ERR_ARG;
  int64_t total = d[0] * d[1] * d[2] * d[3];

  /* step 1: amax over the whole tensor, exact fp32 compares */
  float amax = 0.0f;
  for (int64_t i = 0; i < total; ++i) {
    if (!isfinite(src[i])) return ORC_ERR_NONFINITE;
    float a = fabsf(src[i]);
    if (a > amax) amax = a;
  }
  if (amax_out) *amax_out = amax;
  float amax_used = amax_in ? *amax_in : amax;
  if (!isfinite(amax_used) || amax_used < 0.0f) return ORC_ERR_NONFINITE;

  /* step 2: per-tensor scale */
  float s_t = orc_tensor_scale(fmt, amax_used);
  *s_t_out = s_t;

  double grid[256], grid8[256];
  int cnt = fmt_count(&f), cnt8 = fmt_count(&f8);
  for (int i = 0; i < cnt; ++i) grid[i] = fmt_mag_value(&f, (unsigned)i);
  for (int i = 0; i < cnt8; ++i) grid8[i] = fmt_mag_value(&f8, (unsigned)i);
  double emax = fmt_max(&f);
  unsigned sbit = 1u << (f.ebits + f.mbits);
  int64_t bb = block_bytes(fmt);
  int64_t nblk = orc_num_blocks(role, d);
  memset(codes, 0, (size_t)(nblk * bb));

  int64_t GA = d[0] / 8, GB = d[1] / 8;
#pragma omp parallel for schedule(static)
  for (int64_t blk = 0; blk < nblk; ++blk) {
    int64_t gb = blk % GB, ga = (blk / GB) % GA, s = blk / (GA * GB);
    int64_t s1 = s % d[3], s0 = s / d[3];
    float x[64];
    float amax_b = 0.0f;
    for (int i = 0; i < 64; ++i) {
      int64_t a = ga * 8 + i / 8, b = gb * 8 + i % 8; /* in-block [a][b], b fastest */
      x[i] = src[src_index(layout, d, a, b, s0, s1)];
      if (fabsf(x[i]) > amax_b) amax_b = fabsf(x[i]);
    }
    /* step 3: block scale, nearest E4M3 to amax_b / (maxB_ef * T_scale) */
    unsigned bs_code = 0;
    if (s_t > 0.0f) bs_code = round_mag(grid8, cnt8, (double)amax_b / (emax * (double)s_t));
    double bs = grid8[bs_code];
    scales[blk] = (uint8_t)bs_code;
    /* step 4: element codes, nearest grid value to x / (B_scale * T_scale)
     * (stochastic: one of the two grid values around it, see sr_round_mag) */
    uint8_t *out = codes + blk * bb;
    for (int i = 0; i < 64; ++i) {
      unsigned mag = 0;
      if (bs > 0.0) {
        if (stochastic)
          mag = sr_round_mag(grid, cnt, fabsf(x[i]), (float)bs, s_t, philox_word(seed, blk * 64 + i));
        else
          mag = round_mag(grid, cnt, fabs((double)x[i]) / (bs * (double)s_t));
      }
      put_code(fmt, out, i, mag | (signbit(x[i]) ? sbit : 0u));
    }
  }
  return ORC_OK;
}

int orc_quantize(const float *src, int layout, int role, int fmt, const int64_t d[4],
                 const float *amax_in, uint8_t *codes, uint8_t *scales,
                 float *s_t_out, float *amax_out) {
  return quantize_impl(src, layout, role, fmt, d, amax_in, codes, scales, s_t_out, amax_out, 0, 0);
}

/* ----------------------------------------------------- stochastic rounding */
/*
 * MicroQonv §III-A lets Round be round-to-nearest or stochastic, and uses
 * stochastic rounding for gradients (paperlayer summary, §III-A).  The pages
 * fix neither the random source nor the precision of the decision; these are
 * the readings taken (the kernels implement the same steps):
 *
 *   random source  Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
 *                  random numbers: as easy as 1, 2, 3", SC 2011), keyed by a
 *                  64-bit seed (low word k0, high word k1); element e of the
 *                  packed tensor (e = block * 64 + in-block index) takes
 *                  output word e % 4 of the counter (e / 4 low, e / 4 high,
 *                  0, 0), and its top 24 bits r.
 *   quotient       q = fl32(|x| / fl32(B_scale * T_scale)): one fp32 product
 *                  and one IEEE fp32 division (the kernel's precision).
 *   decision       q >= maxB_ef: the largest code.  Otherwise lo <= q < hi
 *                  are adjacent grid values (hi - lo is a power of two) and
 *                  the code is hi when r < ((q - lo) / (hi - lo)) * 2^24,
 *                  else lo -- every step exact in fp32, so the probability of
 *                  hi is ceil(2^24 (q - lo) / (hi - lo)) / 2^24: the expected
 *                  code value is q to within 2^-24 of the grid spacing.
 * The block scale stays round-to-nearest (CastE4M3 of §III-A).
 */

/* one Philox4x32 round: two 32x32 -> 64-bit products, then the bijection */
static void philox_round(uint32_t c[4], const uint32_t k[2]) {
  const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
  const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
  const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
  const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
  uint32_t n0 = hi1 ^ c[1] ^ k[0], n1 = lo1, n2 = hi0 ^ c[3] ^ k[1], n3 = lo0;
  c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
}

/* Philox4x32-10: ten rounds, the key bumped by the Weyl constants between them */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]}, k[2] = {key[0], key[1]};
  for (int r = 0; r < 10; ++r) {
    if (r > 0) { k[0] += 0x9E3779B9u; k[1] += 0xBB67AE85u; }
    philox_round(c, k);
  }
  for (int i = 0; i < 4; ++i) out[i] = c[i];
}

static uint32_t philox_word(uint64_t seed, int64_t index) {
  const uint64_t q = (uint64_t)index >> 2;
  const uint32_t ctr[4] = {(uint32_t)q, (uint32_t)(q >> 32), 0u, 0u};
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  return out[index & 3];
}

/* Stochastic magnitude code of |x| for block scale bs and T_scale s_t, from
 * one 32-bit random word (steps above; fp32 arithmetic throughout). */
static unsigned sr_round_mag(const double *grid, int n, float ax, float bs, float s_t, uint32_t word) {
  volatile float d = bs * s_t;   /* fl32 product */
  volatile float q = ax / d;     /* IEEE fp32 division */
  if (!(q > 0.0f)) return 0u;
  if ((double)q >= grid[n - 1]) return (unsigned)(n - 1);
  int lo = 0;
  while ((double)q >= grid[lo + 1]) ++lo;            /* grid[lo] <= q < grid[lo + 1] */
  const float g_lo = (float)grid[lo], g_hi = (float)grid[lo + 1];
  volatile float frac = (q - g_lo) / (g_hi - g_lo);  /* exact: Sterbenz, then a power of two */
  volatile float scaled = frac * 16777216.0f;        /* x 2^24, exact */
  const uint32_t r = word >> 8;                      /* top 24 bits */
  return ((float)r < scaled) ? (unsigned)(lo + 1) : (unsigned)lo;
}

int orc_quantize_sr(const float *src, int layout, int role, int fmt, const int64_t d[4],
                    const float *amax_in, uint64_t seed, uint8_t *codes, uint8_t *scales,
                    float *s_t_out, float *amax_out) {
  return quantize_impl(src, layout, role, fmt, d, amax_in, codes, scales, s_t_out, amax_out, 1, seed);
}

/* Fake-quantized (dequantized) values, dense fp64: NCHW for activations and
 * gradients, OIHW for weights.  value = code * B_scale * T_scale, exact in fp64. */
int orc_dequantize(const uint8_t *codes, const uint8_t *scales, float s_t, int role, int fmt,
                   const int64_t d[4], double *out) {
  fmt_t f, f8;
  if (!fmt_get(fmt, &f) || !fmt_get(ORC_E4M3, &f8) || !valid_dims(role, d)) return ORC_ERR_ARG;
  unsigned sbit = 1u << (f.ebits + f.mbits);
  int64_t bb = block_bytes(fmt), GA = d[0] / 8, GB = d[1] / 8;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t s0 = 0; s0 < d[2]; ++s0)
    for (int64_t s1 = 0; s1 < d[3]; ++s1)
      for (int64_t ga = 0; ga < GA; ++ga)
        for (int64_t gb = 0; gb < GB; ++gb) {
          int64_t blk = block_index(d, s0, s1, ga, gb);
          double bs = fmt_mag_value(&f8, scales[blk] & 0x7Fu);
          if (scales[blk] & 0x80u) bs = -bs; /* never produced; decoded faithfully */
          for (int i = 0; i < 64; ++i) {
            unsigned c = get_code(fmt, codes + blk * bb, i);
            double v = fmt_mag_value(&f, c & (sbit - 1u)) * bs * (double)s_t;
            if (c & sbit) v = -v;
            int64_t a = ga * 8 + i / 8, b = gb * 8 + i % 8;
            out[src_index(role == ORC_ROLE_WEIGHT ? ORC_OIHW : ORC_NCHW, d, a, b, s0, s1)] = v;
          }
        }
  return ORC_OK;
}

/* ------------------------------------------------------------ convolution */
/*
 * geometry g = {N, Cin, H, W, Cout, Kh, Kw, stride, pad}; cross-correlation
 * with zero padding (deep-learning convention).  Each sum runs in a fixed
 * order in fp64; `absum` receives sum |a*b| of the same terms.
 */
#define G_N g[0]
#define G_CI g[1]
#define G_H g[2]
#define G_W g[3]
#define G_CO g[4]
#define G_KH g[5]
#define G_KW g[6]
#define G_S g[7]
#define G_P g[8]

static int64_t out_h(const int64_t *g) { return (G_H + 2 * G_P - G_KH) / G_S + 1; }
static int64_t out_w(const int64_t *g) { return (G_W + 2 * G_P - G_KW) / G_S + 1; }

/* Y[n][co][ho][wo] = sum_{ci,kh,kw} W[co][ci][kh][kw] * X[n][ci][ho*s+kh-p][wo*s+kw-p] */
static void fwd_one(const double *X, const double *Wt, const int64_t *g, int64_t n, int64_t co,
                    int64_t ho, int64_t wo, double *y, double *ya) {
  double acc = 0.0, aacc = 0.0;
  for (int64_t ci = 0; ci < G_CI; ++ci)
    for (int64_t kh = 0; kh < G_KH; ++kh)
      for (int64_t kw = 0; kw < G_KW; ++kw) {
        int64_t hi = ho * G_S + kh - G_P, wi = wo * G_S + kw - G_P;
        if (hi < 0 || hi >= G_H || wi < 0 || wi >= G_W) continue;
        double p = Wt[((co * G_CI + ci) * G_KH + kh) * G_KW + kw] *
                   X[((n * G_CI + ci) * G_H + hi) * G_W + wi];
        acc += p;
        aacc += fabs(p);
      }
  *y = acc;
  *ya = aacc;
}

/* dX[n][ci][hi][wi] = sum_{co,kh,kw} W[co][ci][kh][kw] * dY[n][co][ho][wo]
 * over the taps with hi = ho*s + kh - p and wi = wo*s + kw - p (the adjoint
 * of fwd_one: "convolving the output gradient with transposed kernels") */
static void dgrad_one(const double *Wt, const double *dY, const int64_t *g, int64_t n, int64_t ci,
                      int64_t hi, int64_t wi, double *y, double *ya) {
  int64_t Ho = out_h(g), Wo = out_w(g);
  double acc = 0.0, aacc = 0.0;
  for (int64_t co = 0; co < G_CO; ++co)
    for (int64_t kh = 0; kh < G_KH; ++kh)
      for (int64_t kw = 0; kw < G_KW; ++kw) {
        int64_t th = hi + G_P - kh, tw = wi + G_P - kw;
        if (th < 0 || tw < 0 || th % G_S != 0 || tw % G_S != 0) continue;
        int64_t ho = th / G_S, wo = tw / G_S;
        if (ho >= Ho || wo >= Wo) continue;
        double p = Wt[((co * G_CI + ci) * G_KH + kh) * G_KW + kw] *
                   dY[((n * G_CO + co) * Ho + ho) * Wo + wo];
        acc += p;
        aacc += fabs(p);
      }
  *y = acc;
  *ya = aacc;
}

/* dW[co][ci][kh][kw] = sum_{n,ho,wo} dY[n][co][ho][wo] * X[n][ci][ho*s+kh-p][wo*s+kw-p] */
static void wgrad_one(const double *dY, const double *X, const int64_t *g, int64_t co, int64_t ci,
                      int64_t kh, int64_t kw, double *y, double *ya) {
  int64_t Ho = out_h(g), Wo = out_w(g);
  double acc = 0.0, aacc = 0.0;
  for (int64_t n = 0; n < G_N; ++n)
    for (int64_t ho = 0; ho < Ho; ++ho)
      for (int64_t wo = 0; wo < Wo; ++wo) {
        int64_t hi = ho * G_S + kh - G_P, wi = wo * G_S + kw - G_P;
        if (hi < 0 || hi >= G_H || wi < 0 || wi >= G_W) continue;
        double p = dY[((n * G_CO + co) * Ho + ho) * Wo + wo] *
                   X[((n * G_CI + ci) * G_H + hi) * G_W + wi];
        acc += p;
        aacc += fabs(p);
      }
  *y = acc;
  *ya = aacc;
}

/* Full tensors.  Y: (N, Cout, Ho, Wo); dX: (N, Cin, H, W); dW: (Cout, Cin, Kh, Kw). */
void orc_conv_fwd(const double *X, const double *Wt, const int64_t *g, double *Y, double *Ya) {
  int64_t Ho = out_h(g), Wo = out_w(g);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int64_t n = 0; n < G_N; ++n)
    for (int64_t co = 0; co < G_CO; ++co)
      for (int64_t ho = 0; ho < Ho; ++ho)
        for (int64_t wo = 0; wo < Wo; ++wo) {
          int64_t o = ((n * G_CO + co) * Ho + ho) * Wo + wo;
          fwd_one(X, Wt, g, n, co, ho, wo, &Y[o], &Ya[o]);
        }
}

void orc_conv_dgrad(const double *Wt, const double *dY, const int64_t *g, double *dX, double *dXa) {
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int64_t n = 0; n < G_N; ++n)
    for (int64_t ci = 0; ci < G_CI; ++ci)
      for (int64_t hi = 0; hi < G_H; ++hi)
        for (int64_t wi = 0; wi < G_W; ++wi) {
          int64_t o = ((n * G_CI + ci) * G_H + hi) * G_W + wi;
          dgrad_one(Wt, dY, g, n, ci, hi, wi, &dX[o], &dXa[o]);
        }
}

void orc_conv_wgrad(const double *dY, const double *X, const int64_t *g, double *dW, double *dWa) {
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int64_t co = 0; co < G_CO; ++co)
    for (int64_t ci = 0; ci < G_CI; ++ci)
      for (int64_t kh = 0; kh < G_KH; ++kh)
        for (int64_t kw = 0; kw < G_KW; ++kw) {
          int64_t o = ((co * G_CI + ci) * G_KH + kh) * G_KW + kw;
          wgrad_one(dY, X, g, co, ci, kh, kw, &dW[o], &dWa[o]);
        }
}

/* Sampled outputs: idx[] are flat indices into the output tensor's dense
 * layout (same layouts as the full versions). */
void orc_conv_fwd_at(const double *X, const double *Wt, const int64_t *g, const int64_t *idx,
                     int64_t cnt, double *out, double *outa) {
  int64_t Ho = out_h(g), Wo = out_w(g);
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t i = 0; i < cnt; ++i) {
    int64_t o = idx[i];
    int64_t wo = o % Wo, ho = (o / Wo) % Ho, co = (o / (Wo * Ho)) % G_CO, n = o / (Wo * Ho * G_CO);
    fwd_one(X, Wt, g, n, co, ho, wo, &out[i], &outa[i]);
  }
}

void orc_conv_dgrad_at(const double *Wt, const double *dY, const int64_t *g, const int64_t *idx,
                       int64_t cnt, double *out, double *outa) {
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t i = 0; i < cnt; ++i) {
    int64_t o = idx[i];
    int64_t wi = o % G_W, hi = (o / G_W) % G_H, ci = (o / (G_W * G_H)) % G_CI, n = o / (G_W * G_H * G_CI);
    dgrad_one(Wt, dY, g, n, ci, hi, wi, &out[i], &outa[i]);
  }
}

void orc_conv_wgrad_at(const double *dY, const double *X, const int64_t *g, const int64_t *idx,
                       int64_t cnt, double *out, double *outa) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < cnt; ++i) {
    int64_t o = idx[i];
    int64_t kw = o % G_KW, kh = (o / G_KW) % G_KH, ci = (o / (G_KW * G_KH)) % G_CI,
            co = o / (G_KW * G_KH * G_CI);
    wgrad_one(dY, X, g, co, ci, kh, kw, &out[i], &outa[i]);
  }
}
