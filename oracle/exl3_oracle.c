/*
 * CPU oracle for the EXL3 trellis-quantized, Hadamard-rotated linear layer.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library. It shares no code, header,
 * table or constant generator with the CUDA path.
 *
 * What it computes, step by step (plain definitions, FP64, single thread):
 *   1. decode   W[k][n] from the packed trellis tiles (the decode rule below);
 *   2. rot_in   xr = fp16( Hn . (suh o x) ) per 128-block of K, Hn = H/sqrt(128),
 *               H the dense Sylvester matrix H[i][j] = (-1)^popcount(i&j);
 *   3. matmul   z[r][n] = sum_k xr[r][k] W[k][n], summed in FP64, k increasing;
 *   4. rot_out  y = svh o (Hn . z) per 128-block of N.
 * Sources: TensorFold PR #1467 "exl3 cuda: the 27B's EXL3 speed series"
 * (section "What this changes": the rotations rot_in / rot_group, the suh and
 * scales of each member) and PR #1407 item 2 (16x16 tiles grouped in
 * 128-column blocks, n_blocks = stride_k / (bits*8)).
 *
 * Decode rule (the pages name the codebook "mul1" without defining it; this
 * is the build's own QTIP-style rule, written once and followed by both sides):
 *   - a tile is 8*bits uint32 words = a circular stream of L = 256*bits bits,
 *     bit i = (word[i/32] >> (i%32)) & 1 (LSB first);
 *   - weight j (0..255) has the 16-bit state made of stream bits
 *     (j*bits + t) mod L for t = 0..15, bit t of the state = stream bit;
 *   - h = (state * 0x9E3779B1 + 0x7F4A7C15) mod 2^32;
 *   - v = byte0(h) + byte1(h) + byte2(h) + byte3(h)   (0..1020);
 *   - value = (v - 510) / 128   (exact in FP16).
 *   Weight j sits at k_local = 2t + (i&1) + 8*(i>>2), n_local = g + 8*((i>>1)&1)
 *   with lane = j>>3, i = j&7, g = lane>>2, t = lane&3.
 *   Tile (tk, tn) starts at word tk*tile_row_stride + tn*8*bits.
 * PR #1467 (gate 4 paragraph) fixes the window behaviour this rule must show:
 * all-ones words give one value at every width, and a 0xaaaa fill gives two
 * alternating values at odd widths.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#define EXL3O_MUL 0x9E3779B1u
#define EXL3O_ADD 0x7F4A7C15u

/* bit i of a tile's circular stream */
static unsigned stream_bit(const uint32_t *tile, long i) {
  return (tile[i >> 5] >> (i & 31)) & 1u;
}

/* 16-bit state of weight j, built bit by bit from the stream */
uint32_t exl3o_state(const uint32_t *tile, int bits, int j) {
  long L = 256L * bits;
  uint32_t s = 0;
  for (int t = 0; t < 16; t++) {
    long i = ((long)j * bits + t) % L;
    s |= (uint32_t)stream_bit(tile, i) << t;
  }
  return s;
}

/* byte sum of the hashed state: 0..1020 */
int exl3o_code_sum(uint32_t state) {
  uint32_t h = state * EXL3O_MUL + EXL3O_ADD; /* uint32 arithmetic wraps mod 2^32 */
  int v = 0;
  for (int b = 0; b < 4; b++) v += (int)((h >> (8 * b)) & 0xFFu);
  return v;
}

double exl3o_value(uint32_t state) {
  return ((double)exl3o_code_sum(state) - 510.0) / 128.0;
}

void exl3o_position(int j, int *k_local, int *n_local) {
  int lane = j >> 3, i = j & 7, g = lane >> 2, t = lane & 3;
  *n_local = g + 8 * ((i >> 1) & 1);
  *k_local = 2 * t + (i & 1) + 8 * (i >> 2);
}

/* Decode a K x N weight (row-major W[k][n]) whose first tile is at trellis[0].
   A column view passes its advanced pointer and the parent's stride. */
int exl3o_decode(const uint32_t *trellis, long long tile_row_stride, int K, int N, int bits,
                 double *W) {
  if (K % 16 || N % 16 || bits < 1 || bits > 8) return -1;
  for (int tk = 0; tk < K / 16; tk++)
    for (int tn = 0; tn < N / 16; tn++) {
      const uint32_t *tile = trellis + (long long)tk * tile_row_stride + (long long)tn * 8 * bits;
      for (int j = 0; j < 256; j++) {
        int kl, nl;
        exl3o_position(j, &kl, &nl);
        W[(long long)(16 * tk + kl) * N + (16 * tn + nl)] = exl3o_value(exl3o_state(tile, bits, j));
      }
    }
  return 0;
}

/* dense Sylvester Hadamard, entries +-1, row-major 128 x 128 */
void exl3o_hadamard(double *H) {
  for (int i = 0; i < 128; i++)
    for (int j = 0; j < 128; j++) H[i * 128 + j] = (__builtin_popcount((unsigned)(i & j)) & 1) ? -1.0 : 1.0;
}

/* round to the nearest value with `sig` significand bits (round half to even),
   normal exponent floor emin (smallest normal = 2^emin), overflow at `inf_at` */
static double round_to_format(double v, int sig, int emin, double inf_at) {
  if (isnan(v) || isinf(v) || v == 0.0) return v;
  double a = fabs(v);
  if (a >= inf_at) return copysign(INFINITY, v);
  int e;
  frexp(a, &e); /* a in [2^(e-1), 2^e) */
  int qe = e - sig;
  if (qe < emin - sig + 1) qe = emin - sig + 1; /* subnormal quantum */
  double q = ldexp(1.0, qe);
  double r = nearbyint(a / q) * q; /* default rounding mode: nearest, ties to even */
  return copysign(r, v);
}

double exl3o_round_f16(double v) { return round_to_format(v, 11, -14, 65520.0); }
double exl3o_round_bf16(double v) {
  return round_to_format(v, 8, -126, ldexp(2.0 - ldexp(1.0, -8), 127));
}

/* xr[r][k] = fp16( (1/sqrt128) * sum_j H[i][j] * suh[128b+j] * x[r][128b+j] ), k = 128b+i */
int exl3o_rot_in(const double *x, const double *suh, int rows, int K, double *xr) {
  if (K % 128) return -1;
  double *H = malloc(sizeof(double) * 128 * 128);
  if (!H) return -2;
  exl3o_hadamard(H);
  const double c = 1.0 / sqrt(128.0);
  for (int r = 0; r < rows; r++)
    for (int b = 0; b < K / 128; b++)
      for (int i = 0; i < 128; i++) {
        double s = 0.0;
        for (int j = 0; j < 128; j++) {
          long long k = 128LL * b + j;
          s += H[i * 128 + j] * (suh[k] * x[(long long)r * K + k]);
        }
        xr[(long long)r * K + 128LL * b + i] = exl3o_round_f16(c * s);
      }
  free(H);
  return 0;
}

/* z[r][n] = sum_k xr[r][k] * W[k][n], FP64, k in increasing order */
int exl3o_matmul(const double *xr, const double *W, int rows, int K, int N, double *z) {
  for (long long e = 0; e < (long long)rows * N; e++) z[e] = 0.0;
  for (int r = 0; r < rows; r++)
    for (int k = 0; k < K; k++) {
      double a = xr[(long long)r * K + k];
      const double *wrow = W + (long long)k * N;
      double *zrow = z + (long long)r * N;
      for (int n = 0; n < N; n++) zrow[n] += a * wrow[n];
    }
  return 0;
}

/* y[r][128c+i] = svh[128c+i] * (1/sqrt128) * sum_j H[i][j] * z[r][128c+j] */
int exl3o_rot_out(const double *z, const double *svh, int rows, int N, double *y) {
  if (N % 128) return -1;
  double *H = malloc(sizeof(double) * 128 * 128);
  if (!H) return -2;
  exl3o_hadamard(H);
  const double c = 1.0 / sqrt(128.0);
  for (int r = 0; r < rows; r++)
    for (int b = 0; b < N / 128; b++)
      for (int i = 0; i < 128; i++) {
        double s = 0.0;
        for (int j = 0; j < 128; j++) s += H[i * 128 + j] * z[(long long)r * N + 128LL * b + j];
        long long n = 128LL * b + i;
        y[(long long)r * N + n] = svh[n] * (c * s);
      }
  free(H);
  return 0;
}

/* The whole layer: y = svh o Hn( fp16(Hn(suh o x)) . W ). */
int exl3o_linear(const uint32_t *trellis, long long tile_row_stride, int K, int N, int bits,
                 const double *suh, const double *svh, const double *x, int rows, double *y) {
  if (K % 128 || N % 128 || bits < 1 || bits > 8 || rows < 0) return -1;
  double *W = malloc(sizeof(double) * (size_t)K * N);
  double *xr = malloc(sizeof(double) * (size_t)(rows ? rows : 1) * K);
  double *z = malloc(sizeof(double) * (size_t)(rows ? rows : 1) * N);
  int rc = -2;
  if (W && xr && z) {
    rc = exl3o_decode(trellis, tile_row_stride, K, N, bits, W);
    if (!rc) rc = exl3o_rot_in(x, suh, rows, K, xr);
    if (!rc) rc = exl3o_matmul(xr, W, rows, K, N, z);
    if (!rc) rc = exl3o_rot_out(z, svh, rows, N, y);
  }
  free(W);
  free(xr);
  free(z);
  return rc;
}
