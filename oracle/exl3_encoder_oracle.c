/*
 * CPU oracle of the synthetic trellis encoder: targets -> trellis words.
 *
 * TEST INFRASTRUCTURE ONLY (loaded by the tests, the smoke check and the
 * benchmark's CPU legs). It shares no code with the CUDA path; the state
 * value comes from exl3o_code_sum in exl3_oracle.c (same library).
 *
 * The pages quantize with trained checkpoints and never show the encoder; the
 * decode rule is the build's QTIP-style bit-shift trellis (exl3_oracle.c).
 * The encoder follows QTIP (Tseng et al., 2024, "QTIP: Quantization with
 * Trellises and Incoherence Processing"): Viterbi over the shift-register
 * trellis finds the code whose decoded values are closest (sum of squared
 * errors) to the targets, and a tail-biting code is approximated in two
 * passes. Steps, per 16x16 tile (256 weights in stream order j):
 *   - targets are integers on the value grid (units of 1/128, the grid the
 *     decode rule's values lie on), so every cost is an exact integer;
 *   - a state s is a W-bit window (W = 16); moving one weight on shifts
 *     `bits` bits out at the bottom and takes `bits` new bits in at the top:
 *     s' = (s >> bits) | (u << (W - bits)); the predecessors of s' are
 *     p = ((s' & m) << bits) | v, m = 2^(W-bits) - 1, v < 2^bits;
 *   - the cost of state s at weight j is (value(s) - T[j])^2, value(s) =
 *     code_sum(s) - 510; a path's cost is the sum over its 256 states;
 *   - the DP keeps, per state, the cheapest path ending there; among equal
 *     costs the predecessor with the smaller v wins, among equal end costs
 *     the smaller state;
 *   - pass 1: the targets rotated by 128 (T[(j + 128) mod 256]) with any start
 *     and any end; its state at rotated index 128 (the tile's weight 0)
 *     gives the overlap bits c = that state & m;
 *   - pass 2: the targets in order, starts restricted to (s & m) == c and ends
 *     to (s >> bits) == c, which closes the circle: the stream's last state
 *     shifts into its first. Stream bits j*bits .. j*bits+bits-1 are the low
 *     `bits` bits of state j (LSB-first words, as the decode rule reads them).
 * Disallowed starts cost EXL3E_INF (2^30); targets are clamped to
 * [-1024, 1023], so a valid path costs at most 256 * 1534^2 < 2^30.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

int exl3o_code_sum(uint32_t state);
void exl3o_position(int j, int *k_local, int *n_local);

#define EXL3E_INF (1LL << 30)

/* Viterbi over a W-bit shift-register trellis, `bits` bits per step, n steps.
 * val[s]: integer value of state s (2^W entries); T[j]: integer targets.
 * constrain = 0: any start, any end; 1: starts with (s & m) == c, ends with
 * (s >> bits) == c. Writes the best path's states to states[0..n-1] and
 * returns its cost (>= EXL3E_INF when no allowed path exists). */
long long exl3o_viterbi(int W, int bits, int n, const int *val, const int *T, int constrain, uint32_t c,
                        uint32_t *states) {
  if (W < 2 || W > 16 || bits < 1 || bits >= W || n < 1) return -1;
  const uint32_t S = 1u << W, m = (1u << (W - bits)) - 1u, nv = 1u << bits;
  long long *cost = malloc(sizeof(long long) * S), *next = malloc(sizeof(long long) * S);
  unsigned char *dec = malloc((size_t)n * (S >> bits));
  if (!cost || !next || !dec) {
    free(cost);
    free(next);
    free(dec);
    return -2;
  }
  for (uint32_t s = 0; s < S; s++) {
    long long d = (long long)(val[s] - T[0]) * (val[s] - T[0]);
    cost[s] = (!constrain || (s & m) == c) ? d : EXL3E_INF;
  }
  for (int j = 1; j < n; j++) {
    /* best predecessor of each group P of states sharing their low W-bits bits */
    for (uint32_t P = 0; P < (S >> bits); P++) {
      long long best = cost[P << bits];
      unsigned bv = 0;
      for (unsigned v = 1; v < nv; v++)
        if (cost[(P << bits) | v] < best) {
          best = cost[(P << bits) | v];
          bv = v;
        }
      dec[(size_t)j * (S >> bits) + P] = (unsigned char)bv;
      for (uint32_t u = 0; u < nv; u++) {
        const uint32_t s = P | (u << (W - bits));
        const long long d = (long long)(val[s] - T[j]) * (val[s] - T[j]);
        next[s] = best + d;
      }
    }
    long long *t = cost;
    cost = next;
    next = t;
  }
  uint32_t best_s = 0;
  long long best = -1;
  for (uint32_t s = 0; s < S; s++) {
    if (constrain && (s >> bits) != c) continue;
    if (best < 0 || cost[s] < best) {
      best = cost[s];
      best_s = s;
    }
  }
  states[n - 1] = best_s;
  for (int j = n - 1; j > 0; j--) {
    const uint32_t P = states[j] & m;
    states[j - 1] = (P << bits) | dec[(size_t)j * (S >> bits) + P];
  }
  free(cost);
  free(next);
  free(dec);
  return best;
}

/* One tile: 256 grid targets in stream order -> 8*bits words. Returns the
 * squared error of the code (sum over the tile, in grid units^2). */
long long exl3o_encode_tile(const int *T, int bits, const int *val, uint32_t *words) {
  int R[256];
  uint32_t st[256];
  for (int j = 0; j < 256; j++) R[j] = T[(j + 128) % 256];
  if (exl3o_viterbi(16, bits, 256, val, R, 0, 0, st) < 0) return -1;
  const uint32_t m = (1u << (16 - bits)) - 1u;
  const uint32_t c = st[128] & m;
  const long long e = exl3o_viterbi(16, bits, 256, val, T, 1, c, st);
  if (e < 0) return -1;
  memset(words, 0, sizeof(uint32_t) * 8 * bits);
  for (int j = 0; j < 256; j++)
    for (int t = 0; t < bits; t++) {
      const long i = (long)j * bits + t;
      words[i >> 5] |= ((st[j] >> t) & 1u) << (i & 31);
    }
  return e;
}

static int clamp_grid(int t) { return t < -1024 ? -1024 : (t > 1023 ? 1023 : t); }

/* A K x N weight of grid targets (row-major, units of 1/128) -> trellis words
 * in the tile layout of the decode rule (tile (tk, tn) at word
 * tk*(N/16)*8*bits + tn*8*bits). *sq_err gets the total squared error in grid
 * units^2. Tiles [tile0, tile0 + ntiles) of the row-major tile order only
 * (ntiles <= 0: all). */
int exl3o_encode(const int16_t *Tgrid, int K, int N, int bits, long long tile0, long long ntiles, uint32_t *trellis,
                 long long *sq_err) {
  if (K % 16 || N % 16 || bits < 1 || bits > 8) return -1;
  int *val = malloc(sizeof(int) * 65536);
  if (!val) return -2;
  for (uint32_t s = 0; s < 65536; s++) val[s] = exl3o_code_sum(s) - 510;
  const long long TN = N / 16, tiles = (long long)(K / 16) * TN;
  const long long t1 = ntiles > 0 && tile0 + ntiles < tiles ? tile0 + ntiles : tiles;
  long long total = 0;
  for (long long tile = tile0; tile < t1; tile++) {
    const long long tk = tile / TN, tn = tile % TN;
    int T[256];
    for (int j = 0; j < 256; j++) {
      int kl, nl;
      exl3o_position(j, &kl, &nl);
      T[j] = clamp_grid(Tgrid[(16 * tk + kl) * (long long)N + 16 * tn + nl]);
    }
    const long long e = exl3o_encode_tile(T, bits, val, trellis + tk * TN * 8 * bits + tn * 8 * bits);
    if (e < 0) {
      free(val);
      return -3;
    }
    total += e;
  }
  if (sq_err) *sq_err = total;
  free(val);
  return 0;
}
