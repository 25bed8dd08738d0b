/* Seeded synthetic inputs for the fixed-point decoder: weight bytes, row scales, norm
 * weights, prompt ids and test vectors.
 *
 * This module draws random integers and nothing else.  It holds none of the forward
 * pass's arithmetic; both the CPU oracle and the GPU library consume what it writes.
 *
 * Generator: every (tensor, row) pair gets its own xorshift64* stream, the generator the
 * curta-core page gives for sampling ("The inference core", section "Sampling"):
 *     x ^= x >> 12; x ^= x << 25; x ^= x >> 27; out = x * 0x2545F4914F6CDD1D  (mod 2^64)
 * with the rule that a zero state starts at 0x9E3779B97F4A7C15.  The stream's first
 * state is splitmix64 of (base seed, tensor id, row), so rows can be drawn in parallel.
 */
#include <stdint.h>
#include <stddef.h>

#define XS_MULT 0x2545F4914F6CDD1Dull
#define XS_ZERO_SEED 0x9E3779B97F4A7C15ull

static uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* One xorshift64* step: advances *state and returns the scrambled output. */
uint64_t synth_xs64s_next(uint64_t* state) {
  uint64_t x = *state;
  if (x == 0) x = XS_ZERO_SEED;
  x ^= x >> 12;
  x ^= x << 25;
  x ^= x >> 27;
  *state = x;
  return x * XS_MULT;
}

uint64_t synth_stream_seed(uint64_t base, uint32_t tensor, uint64_t row) {
  uint64_t s = splitmix64(base ^ ((uint64_t)tensor << 40));
  s = splitmix64(s ^ row);
  return s ? s : XS_ZERO_SEED;
}

/* rows x cols uniform bytes 0..255, row r at out + r * pitch; bytes cols..pitch-1 are
 * left untouched.  Each 64-bit output yields eight bytes, lowest byte first. */
void synth_bytes(uint8_t* out, uint64_t rows, uint64_t cols, uint64_t pitch, uint64_t base,
                 uint32_t tensor) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < (int64_t)rows; ++r) {
    uint64_t st = synth_stream_seed(base, tensor, (uint64_t)r);
    uint8_t* row = out + (uint64_t)r * pitch;
    uint64_t c = 0;
    while (c < cols) {
      uint64_t v = synth_xs64s_next(&st);
      for (int b = 0; b < 8 && c < cols; ++b, ++c) row[c] = (uint8_t)(v >> (8 * b));
    }
  }
}

/* n values uniform in [lo, hi] (inclusive, hi >= lo), one stream per block of 4096. */
static uint64_t draw_range(uint64_t* st, uint64_t span_minus_1) {
  uint64_t v = synth_xs64s_next(st);
  if (span_minus_1 == ~0ull) return v;
  return v % (span_minus_1 + 1);
}

void synth_u32_range(uint32_t* out, uint64_t n, uint64_t base, uint32_t tensor, uint32_t lo,
                     uint32_t hi) {
  uint64_t blocks = (n + 4095) / 4096;
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < (int64_t)blocks; ++b) {
    uint64_t st = synth_stream_seed(base, tensor, (uint64_t)b);
    uint64_t end = ((uint64_t)b + 1) * 4096 < n ? ((uint64_t)b + 1) * 4096 : n;
    for (uint64_t i = (uint64_t)b * 4096; i < end; ++i)
      out[i] = lo + (uint32_t)draw_range(&st, (uint64_t)(hi - lo));
  }
}

void synth_i64_range(int64_t* out, uint64_t n, uint64_t base, uint32_t tensor, int64_t lo,
                     int64_t hi) {
  uint64_t blocks = (n + 4095) / 4096;
  uint64_t span = (uint64_t)hi - (uint64_t)lo;
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < (int64_t)blocks; ++b) {
    uint64_t st = synth_stream_seed(base, tensor, (uint64_t)b);
    uint64_t end = ((uint64_t)b + 1) * 4096 < n ? ((uint64_t)b + 1) * 4096 : n;
    for (uint64_t i = (uint64_t)b * 4096; i < end; ++i)
      out[i] = (int64_t)((uint64_t)lo + draw_range(&st, span));
  }
}
