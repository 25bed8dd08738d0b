// Internal definitions shared by the libck translation units (device helpers, the state
// layout, the device model layout and the kernel parameter blocks).
#pragma once
#include <cstddef>
#include <cstdint>
#include <algorithm>
#include <cmath>
#include <climits>
#include <cuda_runtime.h>

#include "../../include/ck.h"

namespace ck {

// ------------------------------------------------------------------ state header offsets
constexpr uint32_t kHeaderBytes = 256;
constexpr uint32_t kHPhase = 8, kHPosition = 12, kHNPrompt = 16, kHMaxTok = 20, kHCache = 24,
                   kHGenerated = 28, kHFlags = 32, kHTemp = 36, kHError = 40, kHLastTok = 44,
                   kHSeed = 48, kHTurns = 56, kHErrKey = 64, kHMaxLogit = 72, kHConfig = 80,
                   kHExpSum = 112, kHDraw = 120;
constexpr uint32_t kMaxTemperature = 16u << 16;       // 16 with 16 fraction bits
constexpr unsigned long long kZeroSeedState = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kNoError = ~0ull;

struct StateLayout {
  uint64_t prompt, out, x, xb, q, o, y, h, logits, scores, k, v, size;
  uint32_t cache;
};

inline uint64_t align256(uint64_t n) { return (n + 255) & ~255ull; }

inline StateLayout state_layout(const ck_config& c, uint32_t n_prompt, uint32_t max_tokens) {
  const uint64_t kv_dim = (uint64_t)c.dim / c.heads * c.kv_heads;
  const uint64_t cache = (uint64_t)n_prompt + max_tokens - 1;
  StateLayout s;
  uint64_t off = kHeaderBytes;
  auto take = [&](uint64_t bytes) { uint64_t o = off; off = align256(off + bytes); return o; };
  s.prompt = take(4ull * n_prompt);
  s.out = take(4ull * max_tokens);
  s.x = take(8ull * c.dim);
  s.xb = take(8ull * c.dim);
  s.q = take(8ull * c.dim);
  s.o = take(8ull * c.dim);
  s.y = take(8ull * c.dim);
  s.h = take(8ull * c.hidden);
  s.logits = take(8ull * c.vocab);
  // attention scores and library scratch: max(heads * cache, 1024 * (head + 2) + 2048) words
  const uint64_t hd = c.dim / c.heads;
  const uint64_t words = std::max<uint64_t>((uint64_t)c.heads * cache, 1024 * (hd + 2) + 2048);
  s.scores = take(8ull * words);
  s.k = take(4ull * c.layers * cache * kv_dim);
  s.v = take(4ull * c.layers * cache * kv_dim);
  s.size = off;
  s.cache = (uint32_t)cache;
  return s;
}

// Device-side view of one state header field.
template <typename T>
__device__ __forceinline__ T& hdr(uint8_t* st, uint32_t off) {
  return *reinterpret_cast<T*>(st + off);
}
template <typename T>
__device__ __forceinline__ T hdr_ld(const uint8_t* st, uint32_t off) {
  return *reinterpret_cast<const T*>(st + off);
}

__host__ __device__ inline uint64_t err_key(uint32_t pos, uint32_t layer, uint32_t phase,
                                            uint32_t elem) {
  return ((uint64_t)pos << 44) | ((uint64_t)layer << 32) | ((uint64_t)phase << 24) | elem;
}

// ------------------------------------------------------------------ integer helpers

__host__ __device__ inline uint64_t mulhi_u64(uint64_t a, uint64_t b) {
#ifdef __CUDA_ARCH__
  return __umul64hi(a, b);
#else
  return (uint64_t)(((unsigned __int128)a * b) >> 64);
#endif
}

// Single-precision approximations of 1/x and 1/sqrt(x) (a few units in the last place; the
// hardware's approximate instructions on the device).  The integer routines below only use
// them as estimates and correct every result exactly.
__host__ __device__ inline float rcp_estimate(float x) {
#ifdef __CUDA_ARCH__
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
#else
  return 1.0f / x;
#endif
}
__host__ __device__ inline float rsqrt_estimate(float x) {
#ifdef __CUDA_ARCH__
  float r;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
#else
  return 1.0f / sqrtf(x);
#endif
}

// floor(sqrt(v)) for any u64: an estimate r = v / sqrt(v) in single precision (within about
// 2^-21 of the root, so within 2^11 of it), one Newton step on the exact residual v - r^2
// (a 64-bit value that fits: |v - r^2| < 2^44), then exact integer corrections.  A short
// dependent chain: it sits on the normalization's critical path.
__host__ __device__ inline uint64_t isqrt_u64(uint64_t v) {
  if (v == 0) return 0;
  const float fv = (float)v, y = rsqrt_estimate(fv);
  float fr = fv * y;
  if (fr > 4294967295.0f) fr = 4294967295.0f;
  uint64_t r = (uint64_t)fr;
  if (r > 0xFFFFFFFFull) r = 0xFFFFFFFFull;
  const int64_t e = (int64_t)(v - r * r);
  int64_t t = (int64_t)r + (int64_t)((float)e * (0.5f * y));
  if (t < 0) t = 0;
  if (t > 0xFFFFFFFFll) t = 0xFFFFFFFFll;
  r = (uint64_t)t;
  while (r * r > v) --r;
  while (r < 0xFFFFFFFFull && (r + 1) * (r + 1) <= v) ++r;
  return r;
}

// Division of a u64 by an invariant divisor d (1 <= d < 2^32) with one high multiply,
// after Granlund and Montgomery, "Division by Invariant Integers using Multiplication"
// (PLDI 1994), unsigned case with N = 64: l = ceil(log2 d),
// m = floor(2^64 (2^l - d) / d) + 1, q = (t + ((n - t) >> min(l,1))) >> max(l-1,0) with
// t = mulhi(m, n).
struct InvDiv {
  uint64_t m;
  uint32_t sh1, sh2;
};

__host__ __device__ inline InvDiv make_invdiv(uint32_t d) {
  uint32_t l = 0;
  while (l < 32 && (1ull << l) < (uint64_t)d) ++l;
  const uint64_t a = (1ull << l) - d;  // a < d < 2^32
  // floor(a * 2^64 / d) in two 64/32 steps: both partial quotients are below 2^32
  const uint64_t hi = (a << 32) / d;
  const uint64_t rem = (a << 32) - hi * d;
  const uint64_t lo = (rem << 32) / d;
  InvDiv D;
  D.m = ((hi << 32) | lo) + 1;
  D.sh1 = l < 1 ? l : 1;
  D.sh2 = l > 0 ? l - 1 : 0;
  return D;
}

// floor(n / d) for 1 <= d < 2^32 and n < d * 2^32 (the quotient fits 32 bits): an estimate
// from a single-precision reciprocal, one refinement on the exact remainder, then exact
// integer corrections (both remainders are taken modulo 2^64 and read as signed: their true
// values are far inside the signed range).  Two of these build the reciprocal below in a few
// dozen operations instead of two 64-bit divisions.
__host__ __device__ inline uint64_t div_small_quotient(uint64_t n, uint32_t d) {
  const float rcp = rcp_estimate((float)d);
  uint64_t q = (uint64_t)((float)n * rcp);      // within about 2^10 of the quotient
  if (q > 0xFFFFFFFFull) q = 0xFFFFFFFFull;
  int64_t r = (int64_t)(n - q * d);             // |r| < 2^43
  q = (uint64_t)((int64_t)q + (int64_t)floorf((float)r * rcp));
  r = (int64_t)(n - q * d);                     // within a few d of [0, d)
  while (r < 0) { --q; r += d; }
  while (r >= (int64_t)d) { ++q; r -= d; }
  return q;
}

// floor(num / z) for 1 <= z and a quotient below 2^32 (the probabilities: num = e << 24 with
// e <= z), from rz, an estimate of 1 / z: two estimated steps on exact remainders, then exact
// corrections.  The remainders are taken modulo 2^64 and read as signed; they stay far inside
// that range while num < 2^62.
__host__ __device__ inline uint64_t div_by_estimate(uint64_t num, uint64_t z, float rz) {
  uint64_t q = (uint64_t)((float)num * rz);
  if (q > 0xFFFFFFFFull) q = 0xFFFFFFFFull;
  int64_t r = (int64_t)(num - q * z);
  q = (uint64_t)((int64_t)q + (int64_t)floorf((float)r * rz));
  r = (int64_t)(num - q * z);
  while (r < 0) { --q; r += (int64_t)z; }
  while (r >= (int64_t)z) { ++q; r -= (int64_t)z; }
  return q;
}

// make_invdiv with the two 64-by-32 steps done by div_small_quotient and l = ceil(log2 d)
// from a count of leading zeros.
__host__ __device__ inline InvDiv make_invdiv_fast(uint32_t d) {
#ifdef __CUDA_ARCH__
  const uint32_t l = d <= 1 ? 0u : 32u - (uint32_t)__clz((int)(d - 1));
#else
  const uint32_t l = d <= 1 ? 0u : 32u - (uint32_t)__builtin_clz(d - 1);
#endif
  const uint64_t a = (1ull << l) - d;  // a < d < 2^32
  const uint64_t hi = div_small_quotient(a << 32, d);
  const uint64_t rem = (a << 32) - hi * d;
  const uint64_t lo = div_small_quotient(rem << 32, d);
  InvDiv D;
  D.m = ((hi << 32) | lo) + 1;
  D.sh1 = l < 1 ? l : 1;
  D.sh2 = l > 0 ? l - 1 : 0;
  return D;
}

__host__ __device__ inline uint64_t udiv_inv(uint64_t n, const InvDiv& D) {
  const uint64_t t = mulhi_u64(D.m, n);
  return (t + ((n - t) >> D.sh1)) >> D.sh2;
}

// Signed division truncating toward zero.
__host__ __device__ inline int64_t sdiv_trunc(int64_t n, const InvDiv& D) {
  const uint64_t mag = n < 0 ? 0 - (uint64_t)n : (uint64_t)n;
  const uint64_t q = udiv_inv(mag, D);
  return n < 0 ? (int64_t)(0 - q) : (int64_t)q;
}

__host__ __device__ inline int64_t wmul(int64_t a, int64_t b) {
  return (int64_t)((uint64_t)a * (uint64_t)b);
}
__host__ __device__ inline int64_t wadd(int64_t a, int64_t b) {
  return (int64_t)((uint64_t)a + (uint64_t)b);
}

// The SiLU table lookup ("Lookup tables": 16 or more returns itself, -16 or less zero,
// otherwise entry (x + 16) >> 9).
__device__ __forceinline__ int64_t silu_lookup(int64_t g, const int32_t* tab) {
  const int64_t sixteen = (int64_t)16 << 16;
  if (g >= sixteen) return g;
  if (g <= -sixteen) return 0;
  return (int64_t)__ldg(tab + ((g + sixteen) >> 9));
}

// dp4a with the first operand's bytes unsigned and the second's signed.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ bool fits_i32(int64_t v) { return v >= INT32_MIN && v <= INT32_MAX; }

// Word of element e (0 <= e < kv_dim) of position pos's key or value vector in one layer's
// cache of `cache` positions: head-major, [kv head][position][head element], so one head's
// keys over all positions are one contiguous run.
__host__ __device__ inline size_t cache_word(uint32_t e, uint32_t pos, uint32_t hd, uint32_t cache) {
  return ((size_t)(e / hd) * cache + pos) * hd + e % hd;
}

// First failing cache store wins: the smallest (position, layer, phase, element) key.
__device__ __forceinline__ void record_error(uint8_t* st, uint64_t key) {
  atomicMin(reinterpret_cast<unsigned long long*>(st + kHErrKey), (unsigned long long)key);
}

// Rotation of the pair (a, b) by (cos, sin) with 24 fractional bits, products wrapping.
__device__ __forceinline__ void rotate_pair(int64_t a, int64_t b, int32_t c, int32_t s, int64_t& a2,
                                            int64_t& b2) {
  a2 = (int64_t)((uint64_t)wmul(a, c) - (uint64_t)wmul(b, s)) >> 24;
  b2 = wadd(wmul(a, s), wmul(b, c)) >> 24;
}

// ------------------------------------------------------------------ device model

// Device layout of every model matrix ("column groups").  Rows are padded with zero bytes to
// a multiple of 128 columns, and the columns are cut into groups of 128.  Group g holds, row
// after row, each row's 128 bytes of that group; within them, the row's 16-byte chunk j
// (columns 128g + 16j ..) sits at position j ^ (row & 7).  A block of consecutive rows of
// one group is one contiguous run of memory, so a CTA can copy a rectangle of rows x 128
// columns with one bulk copy, and the rotation of the chunks by the row index lets 32 lanes
// that read the same column chunk of 32 consecutive rows from shared memory hit all banks.
constexpr uint32_t kGroupCols = 128;

__host__ __device__ inline uint32_t pad128(uint32_t n) { return (n + 127u) & ~127u; }

// Byte offset of (row r, column c) in a matrix of `rows` rows in column-group layout.
__host__ __device__ inline uint64_t grouped_offset(uint32_t rows, uint32_t r, uint32_t c) {
  const uint32_t g = c >> 7, j = (c >> 4) & 7u;
  return ((uint64_t)g * rows + r) * kGroupCols + ((j ^ (r & 7u)) << 4) + (c & 15u);
}

struct DevLayer {
  const uint8_t* wqkv;   // [dim + 2 kv_dim][pitch_d]: Wq rows, then Wk, then Wv
  const uint32_t* sqkv;
  const uint8_t* wo;     // [dim][pitch_d]
  const uint32_t* so;
  const uint8_t* w13;    // [2 hidden][pitch_d]: gate row j at 2j, up row j at 2j+1
  const uint32_t* s13;
  const uint8_t* w2;     // [dim][pitch_h]
  const uint32_t* s2;
  const int32_t* attn_norm;
  const int32_t* ffn_norm;
};

// ------------------------------------------------------------------ matrow parameters

enum Prologue : int { kProPlain = 0, kProNorm = 1 };
enum Epilogue : int { kEpiStore = 0, kEpiQKV = 1, kEpiSiLU = 2 };

struct MatrowParams {
  const uint8_t* W;
  const uint32_t* scale;
  uint32_t grouped;      // 1: W in column-group layout (model matrices); 0: row-major
  uint32_t pitch;        // bytes per row, multiple of 16 (of 128 when grouped)
  uint32_t rows, cols;
  // prologue: the input vector of `cols` elements
  int pro;
  const int64_t* in;     // plain: the vector; norm: the activations
  // plain, instead of `in`: wrapping sums whose arithmetic >> 24 is the vector (the attention
  // outputs before their shift); block 0 writes the shifted vector to in_out
  const unsigned long long* in_acc;
  int64_t* in_out;
  // plain, instead of `in`: the vector already as eight byte planes (plane k at k * pitch)
  // with per-CTA partial {wrapping sum, OR of |x|} pairs [nparts][2] of the kernel that
  // wrote them; the prologue copies only the planes the vector needs
  const uint8_t* in_planes;
  const unsigned long long* parts_in;
  uint32_t nparts;
  const int64_t* add;    // norm: residual addend (nullptr: none)
  int64_t* res_out;      // norm with addend: where block 0 writes in + add
  const int32_t* norm_w;
  // norm: the sum of the squares of `in`, complete (added up by the kernel that produced
  // `in`); nullptr: the prologue adds it up itself
  const unsigned long long* ss_in;
  // acc_words words to zero after the wait, split over the CTAs (the attention sums the
  // previous kernel has read, for their next use), or nullptr
  unsigned long long* acc_clear;
  uint32_t acc_words;
  // epilogue
  int epi;
  int64_t* out;          // store: y[rows]; QKV: rotated queries [q_rows]; SiLU: h[rows / 2]
  // SiLU, besides `out`: h as eight byte planes (plane k at k * planes_pitch) and this
  // CTA's {wrapping sum, OR of |h|} at parts_out[2 * blockIdx.x], for the next kernel
  uint8_t* planes_out;
  uint32_t planes_pitch;
  unsigned long long* parts_out;
  // store with a residual (the page's phases 11 and 16 moved into the producing kernel):
  // resid_out[r] = resid_in[r] + y[r], and the squares of resid_out added into *ss_out
  const int64_t* resid_in;
  int64_t* resid_out;
  unsigned long long* ss_out;
  uint32_t q_rows, kv_dim, head_dim, layer, cache;
  int32_t* kcache;       // this layer's keys, position 0 (i32 [cache][kv_dim])
  int32_t* vcache;
  const int32_t* rope;   // [context][head/2][2]
  const int32_t* silu_tab;
  uint8_t* state;        // header for position, phase and errors (nullptr: standalone)
};

struct AttnParams {
  uint8_t* state;
  const int64_t* q;      // rotated queries [heads * hd]
  int64_t* o;            // head outputs [heads * hd] (when o_acc is null)
  // not null: every CTA adds its partial weighted sums of values (before the >> 24) into
  // these zeroed words [heads * hd] instead, and the next kernel applies the shift
  unsigned long long* o_acc;
  const int32_t* kcache; // this layer, position 0
  const int32_t* vcache;
  const uint32_t* exp_tab;
  uint32_t heads, kv_heads, head_dim, kv_dim, inv_sqrt, cache, chunk_cap;
};

// The persistent one-position kernel (ck_step.cu).
// One ring slot: column groups of one row panel.  22 KB holds two groups of panels up to 88
// rows (or one of 96) and lets eight slots fit beside the planes, so that all eight
// consumer warps own stages.
constexpr uint32_t kStageBytes = 22528;
constexpr uint32_t kMaxSlots = 8;        // ring slots at most
constexpr uint32_t kPanelRows = 96;      // most rows of one panel (three a lane)
constexpr uint32_t kStepWarps = 8;       // consumer warps

struct StepParams {
  uint8_t* st;
  uint64_t off_prompt, off_out, off_x, off_xb, off_q, off_o, off_y, off_h, off_logits, off_work,
      off_k, off_v;
  uint32_t cache;
  uint32_t dim, hidden, layers, heads, kv_heads, vocab, hd, kv_dim, pitch_d, pitch_h, inv_sqrt;
  uint32_t generating;  // run phases 17-19 after the layers
  uint32_t gh;          // CTAs per attention head
  uint32_t att_full;    // up to this many positions every CTA of a head scores all of them
  uint32_t ns;          // ring slots
  uint32_t pf_bytes;    // how far ahead of the ring fills the producer prefetches into L2
  uint32_t sync_polls;  // polls of a grid or head-group barrier before it gives up (0: the
                        // default limit); waits on the CTA's own copies keep the default
  uint32_t x_bytes;     // planes, row scales and rotary row / attention region
  uint32_t planes_bytes;  // shared memory for byte planes; a phase keeps
                          // min(8, planes_bytes / pitch) planes there, the rest in global
  // work region (offsets from its start); [0, zero_bytes) is cleared before every launch:
  // barrier and abort words, the per-vector sums and the per-head counters
  uint32_t zero_bytes;
  uint32_t off_hsync, off_hfin;  // per-head barrier counters and finish counters
  uint64_t off_part;    // attention maxima and sums [heads*gh][2]
  uint64_t off_cand;    // classifier candidates [grid][2]
  uint64_t off_oacc;    // attention output accumulators [dim] (u64, before the >> 24)
  uint64_t off_vbuf;    // byte planes of the phase inputs: three buffers of 8 x vbuf_pitch
  uint32_t vbuf_pitch;  // bytes per plane slot (the widest padded vector)
  uint32_t x_vslice, x_wslice;  // X region: this block's residual slice (i64) and the next
                                // norm's weights for it (i32), scale_cap entries each
  uint32_t scale_cap;   // most rows any block takes in one matrix
  InvDiv div_dim, div_hidden;  // for the mean of squares
  const DevLayer* layers_tab;
  const uint8_t* embed;
  const uint32_t* embed_scale;
  const uint8_t* cls;
  const uint32_t* cls_scale;
  const int32_t* final_norm;
  const int32_t* rope;
  const uint32_t* exp_tab;
  const int32_t* silu_tab;
};

// ------------------------------------------------------------------ phase 19 above zero
// "Sampling" at a temperature t > 0 (16 fraction bits).  Sum pass: every logit l adds the
// exponential-table entry at min(((m - l) / t) >> 8, 4096), the difference over the
// temperature taken with 16 fraction bits and truncated.  Draw pass: the generator's output
// modulo the sum, walked through the vocabulary in order, subtracting each entry's
// exponential; the entry it falls inside is the token.
constexpr uint32_t kSampleGroups = 1024;  // u64 partial sums a sampling block keeps in smem

// floor(floor(d * 2^16 / t) / 2^8) = floor(256 d / t) for d = m - l >= 0; that reaches the
// cap 4096 exactly when d >= 16 t, and below it 256 d < 2^32.
__device__ __forceinline__ uint32_t sample_exp_index(long long m, long long l, uint32_t t) {
  const unsigned long long d = (unsigned long long)m - (unsigned long long)l;
  if (d >= 16ull * t) return 4096u;
  return ((uint32_t)d << 8) / t;
}

// xorshift64*: the state moves by the three shifts; the output is the state times the
// multiplier modulo 2^64.
__device__ __forceinline__ unsigned long long sample_next(unsigned long long* state) {
  unsigned long long x = *state;
  x ^= x >> 12;
  x ^= x << 25;
  x ^= x >> 27;
  *state = x;
  return x * 0x2545F4914F6CDD1Dull;
}

__device__ __forceinline__ unsigned long long warp_inclusive_scan(unsigned long long v, uint32_t lane) {
#pragma unroll
  for (uint32_t o = 1; o < 32; o <<= 1) {
    const unsigned long long w = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += w;
  }
  return v;
}

struct SampleOut {
  uint32_t token;
  unsigned long long sum, draw, state;  // state: the generator after the draw
};

// The sum and draw passes by nwarps warps of one block (every thread of them calls it, with
// `bar` synchronising exactly those threads).  Logits are read through L2.  The vocabulary is
// cut into chunks of 32 entries and groups of u chunks (at most kSampleGroups groups); gsum
// (shared memory, kSampleGroups words) receives each group's sum.  The result is valid in
// warp 0.
template <class Bar>
__device__ SampleOut block_sample(const long long* logits, uint32_t vocab, long long m, uint32_t t,
                                  const uint32_t* exp_tab, unsigned long long state,
                                  unsigned long long* gsum, uint32_t nwarps, Bar bar) {
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t nchunk = (vocab + 31) / 32;
  const uint32_t u = (nchunk + kSampleGroups - 1) / kSampleGroups;
  const uint32_t ngroup = (nchunk + u - 1) / u;
  for (uint32_t g = warp; g < ngroup; g += nwarps) {
    unsigned long long s = 0;
    const uint32_t c1 = min(g * u + u, nchunk);
    for (uint32_t c = g * u; c < c1; ++c) {
      const uint32_t i = c * 32 + lane;
      if (i < vocab) s += __ldg(exp_tab + sample_exp_index(m, __ldcg(logits + i), t));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) gsum[g] = s;
  }
  bar();
  SampleOut out{0u, 0ull, 0ull, state};
  if (warp != 0) return out;
  // lane j owns groups [j * seg, (j + 1) * seg)
  const uint32_t seg = (ngroup + 31) / 32;
  const uint32_t g0 = min(lane * seg, ngroup), g1 = min(g0 + seg, ngroup);
  unsigned long long own = 0;
  for (uint32_t g = g0; g < g1; ++g) own += gsum[g];
  const unsigned long long inc = warp_inclusive_scan(own, lane);
  const unsigned long long z = __shfl_sync(0xffffffffu, inc, 31);
  unsigned long long r = 0;
  if (lane == 0) {
    r = sample_next(&state) % z;
    out.state = state;
  }
  r = __shfl_sync(0xffffffffu, r, 0);
  // the lane whose groups hold the draw, then the group, then the chunk, then the entry
  const int L = __ffs(__ballot_sync(0xffffffffu, inc > r)) - 1;
  unsigned long long rem = r - __shfl_sync(0xffffffffu, inc - own, L);
  uint32_t gsel = g0;
  if ((int)lane == L) {
    for (uint32_t g = g0; g < g1; ++g) {
      if (rem < gsum[g]) {
        gsel = g;
        break;
      }
      rem -= gsum[g];
    }
  }
  gsel = __shfl_sync(0xffffffffu, gsel, L);
  rem = __shfl_sync(0xffffffffu, rem, L);
  uint32_t token = 0;
  const uint32_t c1 = min(gsel * u + u, nchunk);
  for (uint32_t c = gsel * u; c < c1; ++c) {
    const uint32_t i = c * 32 + lane;
    const unsigned long long e =
        i < vocab ? (unsigned long long)__ldg(exp_tab + sample_exp_index(m, __ldcg(logits + i), t)) : 0ull;
    const unsigned long long ci = warp_inclusive_scan(e, lane);
    const unsigned long long tot = __shfl_sync(0xffffffffu, ci, 31);
    if (rem < tot) {
      token = c * 32 + (uint32_t)(__ffs(__ballot_sync(0xffffffffu, ci > rem)) - 1);
      break;
    }
    rem -= tot;
  }
  out.token = token;
  out.sum = z;
  out.draw = r;
  return out;
}

// ------------------------------------------------------------------ rows of many positions
// The batched kernels (layer-major prefill of one run, or one position of each of many
// runs) take one descriptor per row: the position it computes and where its run keeps it.
struct RowDesc {
  uint8_t* st;                 // the run's state
  uint32_t pos, cache, np;     // position, cache positions, prompt ids
  uint32_t generating;         // phases 17-19 follow the layers
  uint64_t off_prompt, off_out, off_x, off_logits, off_k, off_v;
};

struct PrefillModel {
  ck_config cfg;
  uint32_t head_dim, kv_dim, inv_sqrt, pitch_d, pitch_h;
  const uint8_t* embed;
  const uint32_t* embed_scale;
  const DevLayer* layers;  // host array of the layer table
  const int32_t* rope;
  const uint32_t* exp_tab;
  const int32_t* silu_tab;
  const uint8_t* cls;
  const uint32_t* cls_scale;
  const int32_t* final_norm;
  int num_sms;
};
// Device scratch a chunk of up to `cap` positions needs.
size_t prefill_work_bytes(const PrefillModel& m, uint32_t cap);
// Whether the batched kernels handle this model and cache length.
bool prefill_supported(const PrefillModel& m, uint32_t cache, size_t smem_optin);
cudaError_t configure_prefill(size_t smem_optin);
// Prompt positions pos0 .. pos0+P-1 (none generating) of the state, layer by layer.
cudaError_t enqueue_prefill(const PrefillModel& m, uint8_t* st, const StateLayout& lay, uint32_t pos0,
                            uint32_t P, uint8_t* work, uint32_t cap, cudaStream_t s);
// Copies the 256-byte headers of n states (device pointers) to host_out; synchronizes.
cudaError_t batch_gather_headers(const PrefillModel& m, uint8_t* const* host_states, uint32_t n,
                                 uint8_t* work, uint32_t cap, uint8_t* host_out, cudaStream_t s);
// One position of each of n runs, with phases 17-19 where a row generates, in two parts: the
// descriptors' copy (host_rows) into the scratch, then the kernels, which read every per-row
// value from the descriptors, so that one capture serves many passes of the same row count;
// max_positions bounds every row's pos + 1.
cudaError_t upload_batch_rows(const PrefillModel& m, const RowDesc* host_rows, uint32_t n, uint8_t* work,
                              uint32_t cap, cudaStream_t s);
cudaError_t enqueue_batch_kernels(const PrefillModel& m, uint32_t n, uint32_t max_positions, uint8_t* work,
                                  uint32_t cap, cudaStream_t s);

cudaError_t configure_step(size_t optin, size_t* dynamic_max);
cudaError_t launch_step(const StepParams& p, cudaStream_t s, int grid, size_t smem);
int step_threads();
size_t noalloc_work_bytes();
cudaError_t noalloc_setup(size_t dynamic_max, uint8_t** work);
cudaError_t launch_step_noalloc(const StepParams& p, uint8_t* work, cudaStream_t s, int grid, size_t smem);
int step_blocks_per_sm(size_t smem);
int step_consumer_warps();
size_t step_red_bytes();

// Launchers (stream-ordered; return a cudaError_t).
cudaError_t configure_matrow();     // once per process and device, outside stream capture
cudaError_t configure_attention();
cudaError_t launch_matrow(const MatrowParams& p, cudaStream_t s, int num_sms);
size_t matrow_smem_bytes(uint32_t pitch);
cudaError_t launch_attention(const AttnParams& p, cudaStream_t s, int cluster);

}  // namespace ck
