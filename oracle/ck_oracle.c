/* ORACLE — test infrastructure, not part of the product.
 *
 * A plain, slow, obviously correct CPU restatement of curta-core's integer forward pass
 * (phases 3 to 19, sampling at temperature zero and above, and the tokenizer of phases 0
 * to 2 with the text of generated tokens), written from the page "The inference core"
 * (curta.chat docs).  Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * may load it.  It shares no code with the GPU library: it parses the model artifact and
 * the state layout itself, from the format description.
 *
 * Every function cites the section of that page it follows.  Wrapping arithmetic is done
 * on uint64_t (defined modulo 2^64 in C); ">>" on int64_t is the arithmetic shift (gcc and
 * clang define it so), "/" on int64_t truncates toward zero.
 *
 * Readings where the page is silent (each one is listed with its reason in the design
 * notes):
 *   r1  (acc - 128*sum) * scale wraps in 64 bits (scale zero-extended), then >> 24.
 *   r4  Squares for RMS normalization wrap in 64 bits and are summed as u64, the mean is
 *       the unsigned quotient, the epsilon is added in u64.
 *   r5  x * weight wraps in 64 bits before the truncating division.
 *   r7  Rotary pairs are elements (2j, 2j+1) of each head, table entry [position][j].
 *   r9  Scores: ((q . k) >> 16) * inv_sqrt wraps, then >> 24.
 *   r10 Weighted values: the sum over positions first, then one >> 24.
 *   r13 Ties in the maximum pass keep the lowest index.
 *   r17 The first failing cache store, in program order, ends the turn with error 8.
 *   r24 Merges of equal score: the leftmost pair merges.
 *   r25 The merge scan looks up every adjacent pair, the opening token's included.
 *   r23 The cache keeps each key/value head's words for all positions together:
 *       [layer][kv head][position][head element]; the page fixes no order inside it.
 *   r20 Sampling divides m - l by the temperature into a value with 16 fractional bits,
 *       truncating; the exponential-table index is that value >> 8, capped at 4,096.
 *   r21 The generator state is the seed word (a zero seed stored as its first state); the
 *       state header records the last sum of exponentials and the last draw.
 *
 * Range events: with counting on, every step that the wrap changes (exact integer result
 * outside int64) is counted, so a workload can show that no reading above mattered.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the OpenMP loops over independent matrix rows use (1 without OpenMP). */
int orc_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ range events */

enum {
  EV_MATROW_ACC = 0,  /* sum (b-128) x outside int64 */
  EV_MATROW_SCALE,    /* (acc - 128 sum) * scale outside int64 */
  EV_NORM_SQUARES,    /* sum of squares outside uint64 */
  EV_NORM_PRODUCT,    /* x * weight outside int64 */
  EV_ROTARY,          /* a*c - b*s or a*s + b*c outside int64 */
  EV_SCORE_DOT,       /* q . k outside int64 */
  EV_SCORE_SCALE,     /* (dot >> 16) * inv outside int64 */
  EV_SILU_PRODUCT,    /* silu(g) * u outside int64 */
  EV_RESIDUAL,        /* x + y outside int64 */
  EV_COUNT
};
static uint64_t g_events[EV_COUNT];
static int g_count_events = 0;

void orc_events_reset(int enable) {
  memset(g_events, 0, sizeof(g_events));
  g_count_events = enable;
}
void orc_events_get(uint64_t* out) { memcpy(out, g_events, sizeof(g_events)); }
static void event(int k) {
#pragma omp atomic
  g_events[k]++;
}
static int outside_i64(__int128 v) { return v > (__int128)INT64_MAX || v < (__int128)INT64_MIN; }

/* ------------------------------------------------------------------ scalar steps */

/* Integer square root, floor(sqrt(v)), by the binary digit-by-digit method.
 * ("RMS normalization": "integer square root".) */
uint64_t orc_isqrt(uint64_t v) {
  uint64_t r = 0, bit = 1ull << 62;
  while (bit > v) bit >>= 2;
  while (bit) {
    if (v >= r + bit) {
      v -= r + bit;
      r = (r >> 1) + bit;
    } else {
      r >>= 1;
    }
    bit >>= 2;
  }
  return r;
}

/* Phase 3, "The forward pass, in order": ((byte - 128) * scale) >> 8 per element. */
void orc_embed(const uint8_t* row, uint32_t scale, uint32_t n, int64_t* x) {
  for (uint32_t i = 0; i < n; ++i) x[i] = ((int64_t)row[i] - 128) * (int64_t)scale >> 8;
}

/* "RMS normalization": rms = isqrt(sum(x*x)/n + 42,950), at least 1;
 * y = ((x * w) / rms) >> 8 with the division rounding toward zero. */
void orc_rmsnorm(const int64_t* x, const int32_t* w, uint32_t n, int64_t* y) {
  uint64_t ss = 0;
  unsigned __int128 exact = 0;
  int over = 0;
  for (uint32_t i = 0; i < n; ++i) {
    ss += (uint64_t)x[i] * (uint64_t)x[i];
    if (g_count_events && !over) {
      unsigned __int128 sq = (unsigned __int128)((__int128)x[i] * x[i]);
      exact += sq;
      over = sq > UINT64_MAX || exact > UINT64_MAX;
    }
  }
  if (over) event(EV_NORM_SQUARES);
  uint64_t mean = ss / n;
  uint64_t rms = orc_isqrt(mean + 42950u);
  if (rms < 1) rms = 1;
  for (uint32_t i = 0; i < n; ++i) {
    int64_t p = (int64_t)((uint64_t)x[i] * (uint64_t)(int64_t)w[i]);
    if (g_count_events && outside_i64((__int128)x[i] * w[i])) event(EV_NORM_PRODUCT);
    int64_t q = p / (int64_t)rms;
    y[i] = q >> 8;
  }
}

/* "A matrix row": sum = x[0] + ... once per vector; acc = sum byte[c] * x[c];
 * y = ((acc - 128 * sum) * scale) >> 24, products wrapping in 64 bits. */
void orc_matrow(const uint8_t* W, uint64_t pitch, const uint32_t* scale, uint32_t rows,
                uint32_t cols, const int64_t* x, int64_t* y) {
  uint64_t sum = 0;
  for (uint32_t c = 0; c < cols; ++c) sum += (uint64_t)x[c];
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < (int64_t)rows; ++r) {
    const uint8_t* row = W + (uint64_t)r * pitch;
    uint64_t acc = 0;
    for (uint32_t c = 0; c < cols; ++c) acc += (uint64_t)row[c] * (uint64_t)x[c];
    uint64_t t = acc - 128u * sum;
    t *= (uint64_t)scale[r];
    y[r] = (int64_t)t >> 24;
    if (g_count_events) {
      __int128 ex = 0;
      for (uint32_t c = 0; c < cols; ++c) ex += (__int128)((int)row[c] - 128) * x[c];
      if (outside_i64(ex)) event(EV_MATROW_ACC);
      else if (outside_i64(ex * (__int128)scale[r])) event(EV_MATROW_SCALE);
    }
  }
}

/* "The attention cache": a store succeeds when the value fits 32 bits. */
int orc_fits32(int64_t v) { return v >= INT32_MIN && v <= INT32_MAX; }

/* Phase 8 (reading r7): rotate the pair (a, b) by (cos, sin) with 24 fractional bits. */
void orc_rotate(int64_t a, int64_t b, int32_t c, int32_t s, int64_t* a2, int64_t* b2) {
  uint64_t ac = (uint64_t)a * (uint64_t)(int64_t)c, bs = (uint64_t)b * (uint64_t)(int64_t)s;
  uint64_t as = (uint64_t)a * (uint64_t)(int64_t)s, bc = (uint64_t)b * (uint64_t)(int64_t)c;
  *a2 = (int64_t)(ac - bs) >> 24;
  *b2 = (int64_t)(as + bc) >> 24;
  if (g_count_events && (outside_i64((__int128)a * c - (__int128)b * s) ||
                         outside_i64((__int128)a * s + (__int128)b * c)))
    event(EV_ROTARY);
}

/* Phase 9, "Attention, stage by stage", for one head over p positions.
 * K and V point at the head's first element of position 0; stride is the distance in
 * words between positions.  scores receives the exponentials at the end (p entries). */
void orc_attention_head(const int64_t* q, const int32_t* K, const int32_t* V, uint64_t stride,
                        uint32_t p, uint32_t hd, uint32_t inv, const uint32_t* exp_tab,
                        int64_t* scores, int64_t* out) {
  /* stage 0: scores and the largest score */
  int64_t m = INT64_MIN;
  for (uint32_t t = 0; t < p; ++t) {
    uint64_t dot = 0;
    __int128 ex = 0;
    for (uint32_t i = 0; i < hd; ++i) {
      int64_t k = K[(uint64_t)t * stride + i];
      dot += (uint64_t)q[i] * (uint64_t)k;
      if (g_count_events) ex += (__int128)q[i] * k;
    }
    int64_t s = (int64_t)dot >> 16;
    if (g_count_events) {
      if (outside_i64(ex)) event(EV_SCORE_DOT);
      else if (outside_i64((__int128)s * inv)) event(EV_SCORE_SCALE);
    }
    s = (int64_t)((uint64_t)s * (uint64_t)inv) >> 24;
    scores[t] = s;
    if (s > m) m = s;
  }
  /* stage 1: exponentials of (largest - score); the exact difference is >= 0 and fits u64 */
  uint64_t sum = 0;
  for (uint32_t t = 0; t < p; ++t) {
    uint64_t d = (uint64_t)m - (uint64_t)scores[t];
    uint64_t idx = d >> 8;
    if (idx > 4096) idx = 4096;
    scores[t] = (int64_t)exp_tab[idx];
    sum += exp_tab[idx];
  }
  /* stage 2: probabilities with 24 fractional bits */
  for (uint32_t t = 0; t < p; ++t) scores[t] = (int64_t)(((uint64_t)scores[t] << 24) / sum);
  /* stage 3: weighted values, the sum first, then one shift */
  for (uint32_t j = 0; j < hd; ++j) {
    uint64_t acc = 0;
    for (uint32_t t = 0; t < p; ++t)
      acc += (uint64_t)scores[t] * (uint64_t)(int64_t)V[(uint64_t)t * stride + j];
    out[j] = (int64_t)acc >> 24;
  }
}

/* "Lookup tables", SiLU: 16 or more returns itself, -16 or less returns zero, otherwise
 * the entry (x + 16) >> 9 in fixed point. */
int64_t orc_silu(int64_t g, const int32_t* tab) {
  const int64_t sixteen = (int64_t)16 << 16;
  if (g >= sixteen) return g;
  if (g <= -sixteen) return 0;
  return tab[(g + sixteen) >> 9];
}

/* Phase 14: each gate element through the table, times the up element, >> 16. */
void orc_silu_gate(const int64_t* g, const int64_t* u, uint32_t n, const int32_t* tab, int64_t* h) {
  for (uint32_t i = 0; i < n; ++i) {
    int64_t s = orc_silu(g[i], tab);
    if (g_count_events && outside_i64((__int128)s * u[i])) event(EV_SILU_PRODUCT);
    h[i] = (int64_t)((uint64_t)s * (uint64_t)u[i]) >> 16;
  }
}

/* Phase 19 at temperature zero ("Sampling", maximum pass): the first largest logit. */
uint32_t orc_argmax(const int64_t* logits, uint32_t n) {
  uint32_t best = 0;
  for (uint32_t i = 1; i < n; ++i)
    if (logits[i] > logits[best]) best = i;
  return best;
}

/* "Sampling", the generator: xorshift64* (shifts 12 right, 25 left, 27 right, then the
 * product with 0x2545F4914F6CDD1D mod 2^64).  Advances the state once and returns the
 * output; the shifted value, not the product, is the new state. */
uint64_t orc_xorshift_next(uint64_t* state) {
  uint64_t x = *state;
  x ^= x >> 12;
  x ^= x << 25;
  x ^= x >> 27;
  *state = x;
  return x * 0x2545F4914F6CDD1Dull;
}

/* "Sampling", sum pass: the exponential-table index of a logit l below the largest logit m
 * at temperature t (16 fractional bits, 1 ..= 16 << 16).  The difference m - l, which has
 * 16 fractional bits and is zero or more, is divided by the temperature, truncating, into a
 * value that again has 16 fractional bits; the index is that value >> 8, capped at 4,096,
 * as for every read of the exponential table.  Computed in 128 bits, so nothing wraps. */
uint32_t orc_sample_index(int64_t m, int64_t l, uint32_t t) {
  unsigned __int128 d = (unsigned __int128)((__int128)m - (__int128)l);
  unsigned __int128 scaled = (d << 16) / t;
  unsigned __int128 idx = scaled >> 8;
  return idx > 4096 ? 4096u : (uint32_t)idx;
}

/* "Sampling", draw pass walk: from the remainder r, subtract each entry's exponential in
 * vocabulary order and take the first entry the remainder falls inside. */
uint32_t orc_draw_walk(const uint64_t* e, uint32_t n, uint64_t r) {
  for (uint32_t i = 0; i < n; ++i) {
    if (r < e[i]) return i;
    r -= e[i];
  }
  return n; /* r was not below the sum: no entry */
}

/* Phase 19, "Sampling": the maximum pass, and above temperature zero the sum and draw
 * passes.  gen is the run's generator state (advanced once per draw); m, sum and draw
 * receive the largest logit, the sum of exponentials and the draw (0 at temperature 0). */
uint32_t orc_sample(const int64_t* logits, uint32_t n, uint32_t t, const uint32_t* exp_tab,
                    uint64_t* gen, int64_t* m, uint64_t* sum, uint64_t* draw) {
  uint32_t best = orc_argmax(logits, n);                       /* maximum pass */
  *m = logits[best];
  *sum = 0;
  *draw = 0;
  if (t == 0) return best;
  uint64_t* e = (uint64_t*)malloc(8ull * n);
  uint64_t z = 0;
  for (uint32_t i = 0; i < n; ++i) {                            /* sum pass */
    e[i] = exp_tab[orc_sample_index(*m, logits[i], t)];
    z += e[i];
  }
  uint64_t r = orc_xorshift_next(gen) % z;                      /* draw pass */
  uint32_t chosen = orc_draw_walk(e, n, r);
  free(e);
  *sum = z;
  *draw = r;
  return chosen;
}

static void residual(int64_t* x, const int64_t* y, uint32_t n) {
  for (uint32_t i = 0; i < n; ++i) {
    if (g_count_events && outside_i64((__int128)x[i] + y[i])) event(EV_RESIDUAL);
    x[i] = (int64_t)((uint64_t)x[i] + (uint64_t)y[i]);
  }
}

/* ------------------------------------------------------------------ the state size the
 * page gives ("The resumable state"): text-mode buffers, each at a multiple of 8 bytes. */
static uint64_t up8(uint64_t n) { return (n + 7) & ~7ull; }

uint64_t orc_page_state_size(const uint32_t* cfg, uint32_t prompt_bytes, uint32_t max_tokens) {
  uint64_t dim = cfg[0], hidden = cfg[1], layers = cfg[2], heads = cfg[3], kvh = cfg[4];
  uint64_t vocab = cfg[5], context = cfg[6];
  uint64_t kv_dim = dim / heads * kvh;
  uint64_t cache = (uint64_t)prompt_bytes + max_tokens + 1;
  if (cache > context) cache = context;
  uint64_t n = 128;
  n = up8(n + prompt_bytes);
  n = up8(n + 4ull * (prompt_bytes + 2));
  n = up8(n + 4ull * max_tokens);
  n = up8(n + 128ull * max_tokens);
  n = up8(n + 4 * 8 * dim);
  n = up8(n + 2 * 8 * hidden);
  n = up8(n + 8 * vocab);
  n = up8(n + 8 * cache);
  n = up8(n + 4 * layers * cache * kv_dim);
  n = up8(n + 4 * layers * cache * kv_dim);
  return n;
}

/* ------------------------------------------------------------------ model artifact */

typedef struct {
  const int32_t *attn_norm, *ffn_norm;
  const uint8_t *wq, *wk, *wv, *wo, *w1, *w3, *w2;
  const uint32_t *sq, *sk, *sv, *so, *s1, *s3, *s2;
} orc_layer;

typedef struct {
  uint32_t dim, hidden, layers, heads, kv_heads, vocab, context;
  uint32_t head_dim, kv_dim, inv_sqrt, flags;
  const uint8_t* embed;
  const uint32_t* embed_scale;
  const int32_t* final_norm;
  const uint8_t* cls;
  const uint32_t* cls_scale;
  const int32_t* rope;
  const uint32_t* exp_tab;
  const int32_t* silu_tab;
  orc_layer* layer;
} orc_model;

static uint32_t rd32(const uint8_t* p) { uint32_t v; memcpy(&v, p, 4); return v; }
static uint64_t rd64(const uint8_t* p) { uint64_t v; memcpy(&v, p, 8); return v; }

/* Parses an artifact (format "CKMODEL1", see the library header).  Returns 0, 1 for an
 * invalid configuration or 2 for an invalid format; pointers alias the artifact. */
int orc_model_open(const uint8_t* art, uint64_t len, orc_model** out) {
  *out = NULL;
  if (len < 64 || memcmp(art, "CKMODEL1", 8) != 0) return 2;
  orc_model m;
  memset(&m, 0, sizeof(m));
  m.dim = rd32(art + 8); m.hidden = rd32(art + 12); m.layers = rd32(art + 16);
  m.heads = rd32(art + 20); m.kv_heads = rd32(art + 24); m.vocab = rd32(art + 28);
  m.context = rd32(art + 32); m.inv_sqrt = rd32(art + 36); m.flags = rd32(art + 40);
  uint32_t n_tensors = rd32(art + 44);
  if (!m.dim || !m.hidden || !m.layers || !m.heads || !m.kv_heads || !m.vocab || !m.context) return 1;
  if (m.dim % m.heads || m.heads % m.kv_heads || (m.dim / m.heads) % 2) return 1;
  m.head_dim = m.dim / m.heads;
  m.kv_dim = m.head_dim * m.kv_heads;
  if (n_tensors != 8 + 16 * m.layers || rd64(art + 48) != len) return 2;
  if (64 + 16ull * n_tensors > len) return 2;
  const uint64_t d = m.dim, h = m.hidden, v = m.vocab, kv = m.kv_dim;
  int tied = m.flags & 1;
  uint64_t want[8] = {v * d, 4 * v, 4 * d, tied ? 0 : v * d, tied ? 0 : 4 * v,
                      4ull * m.context * m.head_dim, 4 * 4097, 4 * 4097};
  uint64_t want_layer[16] = {4 * d, d * d, 4 * d, kv * d, 4 * kv, kv * d, 4 * kv, d * d,
                             4 * d, 4 * d, h * d, 4 * h, h * d, 4 * h, d * h, 4 * d};
  if (m.layers > 4096) return 1;
  const uint8_t** ptr = (const uint8_t**)calloc(n_tensors, sizeof(*ptr));
  for (uint32_t i = 0; i < n_tensors; ++i) {
    uint64_t off = rd64(art + 64 + 16 * i), tl = rd64(art + 64 + 16 * i + 8);
    uint64_t expect = i < 8 ? want[i] : want_layer[(i - 8) % 16];
    if (tl != expect || (tl && (off > len || tl > len - off || off % 4))) {
      free(ptr);
      return 2;
    }
    ptr[i] = art + off;
  }
  m.embed = ptr[0];
  m.embed_scale = (const uint32_t*)ptr[1];
  m.final_norm = (const int32_t*)ptr[2];
  m.cls = tied ? m.embed : ptr[3];
  m.cls_scale = tied ? m.embed_scale : (const uint32_t*)ptr[4];
  m.rope = (const int32_t*)ptr[5];
  m.exp_tab = (const uint32_t*)ptr[6];
  m.silu_tab = (const int32_t*)ptr[7];
  m.layer = (orc_layer*)calloc(m.layers, sizeof(orc_layer));
  for (uint32_t l = 0; l < m.layers; ++l) {
    const uint8_t** p = ptr + 8 + 16 * l;
    orc_layer* L = &m.layer[l];
    L->attn_norm = (const int32_t*)p[0];
    L->wq = p[1]; L->sq = (const uint32_t*)p[2];
    L->wk = p[3]; L->sk = (const uint32_t*)p[4];
    L->wv = p[5]; L->sv = (const uint32_t*)p[6];
    L->wo = p[7]; L->so = (const uint32_t*)p[8];
    L->ffn_norm = (const int32_t*)p[9];
    L->w1 = p[10]; L->s1 = (const uint32_t*)p[11];
    L->w3 = p[12]; L->s3 = (const uint32_t*)p[13];
    L->w2 = p[14]; L->s2 = (const uint32_t*)p[15];
  }
  free(ptr);
  *out = (orc_model*)malloc(sizeof(orc_model));
  **out = m;
  return 0;
}

void orc_model_close(orc_model* m) {
  if (m) {
    free(m->layer);
    free(m);
  }
}

/* ------------------------------------------------------------------ state ("CKSTATE1")
 * The ids-mode state of the library header: a 256-byte header, then the buffers, each at
 * a multiple of 256 bytes: prompt ids u32[n_prompt], output tokens u32[max_tokens],
 * x, xb, q, o, y i64[dim], h i64[hidden], logits i64[vocab],
 * scores (work) i64[max(heads*cache, 1024*(head+2)+2048)], K i32[layers][kv heads][cache][head],
 * V i32 likewise (head-major, reading r23). */

enum { H_PHASE = 8, H_POSITION = 12, H_NPROMPT = 16, H_MAXTOK = 20, H_CACHE = 24, H_GENERATED = 28,
       H_FLAGS = 32, H_TEMP = 36, H_ERROR = 40, H_LASTTOK = 44, H_SEED = 48, H_TURNS = 56,
       H_ERRKEY = 64, H_MAXLOGIT = 72, H_CONFIG = 80, H_EXPSUM = 112, H_DRAW = 120 };
enum { PHASE_RUNNING = 3, PHASE_DONE = 20, PHASE_FAILED = 21 };

typedef struct {
  uint64_t prompt, out, x, xb, q, o, y, h, logits, scores, k, v, size;
} orc_layout;

static uint64_t up256(uint64_t n) { return (n + 255) & ~255ull; }

static orc_layout layout_of(const uint32_t* cfg, uint32_t n_prompt, uint32_t max_tokens) {
  uint64_t dim = cfg[0], hidden = cfg[1], layers = cfg[2], heads = cfg[3], kvh = cfg[4];
  uint64_t vocab = cfg[5];
  uint64_t kv_dim = dim / heads * kvh;
  uint64_t cache = (uint64_t)n_prompt + max_tokens - 1;
  orc_layout L;
  uint64_t n = 256;
  L.prompt = n; n = up256(n + 4ull * n_prompt);
  L.out = n; n = up256(n + 4ull * max_tokens);
  L.x = n; n = up256(n + 8 * dim);
  L.xb = n; n = up256(n + 8 * dim);
  L.q = n; n = up256(n + 8 * dim);
  L.o = n; n = up256(n + 8 * dim);
  L.y = n; n = up256(n + 8 * dim);
  L.h = n; n = up256(n + 8 * hidden);
  L.logits = n; n = up256(n + 8 * vocab);
  /* scores / work region: max(heads * cache, 1024 * (head + 2) + 2048) i64 words */
  uint64_t hd = dim / heads;
  uint64_t words = heads * cache > 1024 * (hd + 2) + 2048 ? heads * cache : 1024 * (hd + 2) + 2048;
  L.scores = n; n = up256(n + 8 * words);
  L.k = n; n = up256(n + 4 * layers * cache * kv_dim);
  L.v = n; n = up256(n + 4 * layers * cache * kv_dim);
  L.size = n;
  return L;
}

static void model_cfg(const orc_model* m, uint32_t* cfg) {
  cfg[0] = m->dim; cfg[1] = m->hidden; cfg[2] = m->layers; cfg[3] = m->heads;
  cfg[4] = m->kv_heads; cfg[5] = m->vocab; cfg[6] = m->context;
}

uint64_t orc_state_size(const orc_model* m, uint32_t n_prompt, uint32_t max_tokens) {
  uint32_t cfg[7];
  model_cfg(m, cfg);
  if (n_prompt == 0 || max_tokens == 0) return 0;
  return layout_of(cfg, n_prompt, max_tokens).size;
}

static void wr32(uint8_t* p, uint32_t v) { memcpy(p, &v, 4); }
static void wr64(uint8_t* p, uint64_t v) { memcpy(p, &v, 8); }

/* "The Rust API", init_state, in ids mode: writes a fresh header and the prompt ids.
 * Errors: 4 wrong length, 3 misaligned, 6 invalid prompt / max tokens / temperature,
 * 7 prompt plus max tokens less one above the context. */
int orc_init_state(const orc_model* m, uint8_t* st, uint64_t len, const uint32_t* ids,
                   uint32_t n_ids, uint32_t max_tokens, uint32_t temperature_q16, uint64_t seed,
                   uint32_t flags) {
  if ((uintptr_t)st % 8) return 3;
  if (n_ids == 0 || max_tokens == 0 || max_tokens > m->context) return 6;
  if (temperature_q16 > (16u << 16)) return 6; /* a temperature above 16 */
  for (uint32_t i = 0; i < n_ids; ++i)
    if (ids[i] >= m->vocab) return 6;
  if ((uint64_t)n_ids + max_tokens - 1 > m->context) return 7;
  uint32_t cfg[7];
  model_cfg(m, cfg);
  orc_layout L = layout_of(cfg, n_ids, max_tokens);
  if (len != L.size) return 4;
  memset(st, 0, len);
  memcpy(st, "CKSTATE1", 8);
  wr32(st + H_PHASE, PHASE_RUNNING);
  wr32(st + H_NPROMPT, n_ids);
  wr32(st + H_MAXTOK, max_tokens);
  wr32(st + H_CACHE, n_ids + max_tokens - 1);
  wr32(st + H_FLAGS, flags);
  wr32(st + H_TEMP, temperature_q16);
  wr32(st + H_LASTTOK, 0xFFFFFFFFu);
  wr64(st + H_SEED, seed ? seed : 0x9E3779B97F4A7C15ull); /* a zero seed's first state */
  wr64(st + H_ERRKEY, ~0ull);
  for (int i = 0; i < 7; ++i) wr32(st + H_CONFIG + 4 * i, cfg[i]);
  memcpy(st + L.prompt, ids, 4ull * n_ids);
  return 0;
}

typedef struct {
  uint32_t complete, generated, generated_this_turn, token, work;
  uint32_t err_position, err_layer, err_phase, err_element;
} orc_turn_result;

static uint64_t err_key(uint32_t pos, uint32_t layer, uint32_t phase, uint32_t elem) {
  return ((uint64_t)pos << 44) | ((uint64_t)layer << 32) | ((uint64_t)phase << 24) | elem;
}

/* Index of element j (0 <= j < kv_dim) of position pos's key or value vector in layer l's
 * cache: head-major, [layer][kv head][position][head element] (reading r23). */
static uint64_t cache_index(uint32_t l, uint32_t cache, uint32_t pos, uint32_t j, uint32_t hd,
                            uint32_t kvd) {
  return (uint64_t)l * cache * kvd + ((uint64_t)(j / hd) * cache + pos) * hd + j % hd;
}

/* One position, phases 3 to 16 for every layer, then 17 to 19 where a token is generated
 * ("The forward pass, in order").  Returns 0, or 8 at the first store that does not fit. */
static int run_position(const orc_model* m, uint8_t* st, const orc_layout* L) {
  const uint32_t pos = rd32(st + H_POSITION), n_prompt = rd32(st + H_NPROMPT);
  const uint32_t cache = rd32(st + H_CACHE);
  const uint32_t* prompt = (const uint32_t*)(st + L->prompt);
  uint32_t* out = (uint32_t*)(st + L->out);
  int64_t *x = (int64_t*)(st + L->x), *xb = (int64_t*)(st + L->xb), *q = (int64_t*)(st + L->q);
  int64_t *o = (int64_t*)(st + L->o), *y = (int64_t*)(st + L->y), *hh = (int64_t*)(st + L->h);
  int64_t *logits = (int64_t*)(st + L->logits), *scores = (int64_t*)(st + L->scores);
  int32_t *Kc = (int32_t*)(st + L->k), *Vc = (int32_t*)(st + L->v);
  const uint32_t d = m->dim, hd = m->head_dim, kvd = m->kv_dim, hid = m->hidden;
  int64_t* g = (int64_t*)malloc(8ull * hid * 2);
  int64_t* u = g + hid;
  int64_t* kv = (int64_t*)malloc(8ull * kvd);
  int rc = 0;

  /* phase 3: the token of this position is a prompt id or the last generated token */
  uint32_t tok = pos < n_prompt ? prompt[pos] : out[pos - n_prompt];
  if (tok >= m->vocab) { /* a state edited outside init_state and turn */
    free(g);
    free(kv);
    return 3;
  }
  orc_embed(m->embed + (uint64_t)tok * d, m->embed_scale[tok], d, x);

  for (uint32_t l = 0; l < m->layers && !rc; ++l) {
    const orc_layer* W = &m->layer[l];
    /* element j of this position's key or value vector (reading r23: head-major cache) */
#define KV_AT(C, j) ((C)[cache_index(l, cache, pos, (j), hd, kvd)])
    orc_rmsnorm(x, W->attn_norm, d, xb);                               /* phase 4 */
    orc_matrow(W->wq, d, W->sq, d, d, xb, q);                          /* phase 5 */
    orc_matrow(W->wk, d, W->sk, kvd, d, xb, kv);                       /* phase 6 */
    for (uint32_t j = 0; j < kvd && !rc; ++j) {
      if (!orc_fits32(kv[j])) { rc = 8; wr64(st + H_ERRKEY, err_key(pos, l, 6, j)); }
      else KV_AT(Kc, j) = (int32_t)kv[j];
    }
    if (rc) break;
    orc_matrow(W->wv, d, W->sv, kvd, d, xb, kv);                       /* phase 7 */
    for (uint32_t j = 0; j < kvd && !rc; ++j) {
      if (!orc_fits32(kv[j])) { rc = 8; wr64(st + H_ERRKEY, err_key(pos, l, 7, j)); }
      else KV_AT(Vc, j) = (int32_t)kv[j];
    }
    if (rc) break;
    const int32_t* rope = m->rope + (uint64_t)pos * hd;                /* phase 8 */
    for (uint32_t i = 0; i < d; i += 2) {
      uint32_t j = (i % hd) / 2;
      orc_rotate(q[i], q[i + 1], rope[2 * j], rope[2 * j + 1], &q[i], &q[i + 1]);
    }
    for (uint32_t i = 0; i < kvd && !rc; i += 2) {
      uint32_t j = (i % hd) / 2;
      int64_t a2, b2;
      orc_rotate(KV_AT(Kc, i), KV_AT(Kc, i + 1), rope[2 * j], rope[2 * j + 1], &a2, &b2);
      if (!orc_fits32(a2)) { rc = 8; wr64(st + H_ERRKEY, err_key(pos, l, 8, i)); break; }
      KV_AT(Kc, i) = (int32_t)a2;
      if (!orc_fits32(b2)) { rc = 8; wr64(st + H_ERRKEY, err_key(pos, l, 8, i + 1)); break; }
      KV_AT(Kc, i + 1) = (int32_t)b2;
    }
    if (rc) break;
    const uint32_t group = m->heads / m->kv_heads;                     /* phase 9 */
    for (uint32_t hh_ = 0; hh_ < m->heads; ++hh_) {
      uint32_t kvh = hh_ / group;
      const int32_t* K0 = Kc + cache_index(l, cache, 0, kvh * hd, hd, kvd);
      const int32_t* V0 = Vc + cache_index(l, cache, 0, kvh * hd, hd, kvd);
      orc_attention_head(q + (uint64_t)hh_ * hd, K0, V0, hd, pos + 1, hd, m->inv_sqrt, m->exp_tab,
                         scores + (uint64_t)hh_ * cache, o + (uint64_t)hh_ * hd);
    }
#undef KV_AT
    orc_matrow(W->wo, d, W->so, d, d, o, y);                           /* phase 10 */
    residual(x, y, d);                                                 /* phase 11 */
    orc_rmsnorm(x, W->ffn_norm, d, xb);
    orc_matrow(W->w1, d, W->s1, hid, d, xb, g);                        /* phase 12 */
    orc_matrow(W->w3, d, W->s3, hid, d, xb, u);                        /* phase 13 */
    orc_silu_gate(g, u, hid, m->silu_tab, hh);                         /* phase 14 */
    orc_matrow(W->w2, hid, W->s2, d, hid, hh, y);                      /* phase 15 */
    residual(x, y, d);                                                 /* phase 16 */
  }
  free(g);
  free(kv);
  if (rc) return rc;

  if (pos + 1 >= n_prompt) {                                           /* a generating position */
    orc_rmsnorm(x, m->final_norm, d, xb);                              /* phase 17 */
    orc_matrow(m->cls, d, m->cls_scale, m->vocab, d, xb, logits);      /* phase 18 */
    uint64_t state = rd64(st + H_SEED), z, draw;                       /* phase 19 */
    int64_t mx;
    uint32_t t = orc_sample(logits, m->vocab, rd32(st + H_TEMP), m->exp_tab, &state, &mx, &z,
                            &draw);
    uint32_t gen = rd32(st + H_GENERATED);
    out[gen] = t;
    wr32(st + H_GENERATED, gen + 1);
    wr32(st + H_LASTTOK, t);
    wr64(st + H_MAXLOGIT, (uint64_t)mx);
    wr64(st + H_SEED, state);
    wr64(st + H_EXPSUM, z);
    wr64(st + H_DRAW, draw);
    if (gen + 1 == rd32(st + H_MAXTOK) || ((rd32(st + H_FLAGS) & 1) && (t == 1 || t == 2)))
      wr32(st + H_PHASE, PHASE_DONE);
  }
  wr32(st + H_POSITION, pos + 1);
  return 0;
}

/* "The Rust API", turn: runs up to n_positions positions of the run.  Errors: 3 for a
 * state that does not fit the model or is complete, 8 for a cache store that does not
 * fit (the state is then marked failed). */
int orc_turn(const orc_model* m, uint8_t* st, uint64_t len, uint32_t n_positions,
             orc_turn_result* res) {
  memset(res, 0, sizeof(*res));
  res->token = 0xFFFFFFFFu;
  if ((uintptr_t)st % 8 || len < 256 || memcmp(st, "CKSTATE1", 8) != 0) return 3;
  uint32_t cfg[7];
  model_cfg(m, cfg);
  for (int i = 0; i < 7; ++i)
    if (rd32(st + H_CONFIG + 4 * i) != cfg[i]) return 3;
  const uint32_t n_prompt = rd32(st + H_NPROMPT), max_tokens = rd32(st + H_MAXTOK);
  if (!n_prompt || !max_tokens || (uint64_t)n_prompt + max_tokens - 1 > m->context) return 3;
  orc_layout L = layout_of(cfg, n_prompt, max_tokens);
  if (len != L.size || rd32(st + H_CACHE) != n_prompt + max_tokens - 1) return 3;
  if (rd32(st + H_PHASE) != PHASE_RUNNING) return 3;
  const uint32_t pos = rd32(st + H_POSITION);
  if (pos >= n_prompt + max_tokens - 1) return 3;
  /* tokens generated so far equal the generating positions already run */
  if (rd32(st + H_GENERATED) != (pos + 1 > n_prompt ? pos + 1 - n_prompt : 0)) return 3;
  int rc = 0;
  uint32_t gen0 = rd32(st + H_GENERATED);
  for (uint32_t i = 0; i < n_positions; ++i) {
    if (rd32(st + H_PHASE) != PHASE_RUNNING) break;
    uint32_t before = rd32(st + H_GENERATED);
    rc = run_position(m, st, &L);
    res->work++;
    if (rc) {
      wr32(st + H_PHASE, PHASE_FAILED);
      wr32(st + H_ERROR, (uint32_t)rc);
      break;
    }
    if (rd32(st + H_GENERATED) != before) res->token = rd32(st + H_LASTTOK);
  }
  wr64(st + H_TURNS, rd64(st + H_TURNS) + 1);
  res->generated = rd32(st + H_GENERATED);
  res->generated_this_turn = res->generated - gen0;
  res->complete = rd32(st + H_PHASE) != PHASE_RUNNING;
  uint64_t key = rd64(st + H_ERRKEY);
  if (key != ~0ull) {
    res->err_position = (uint32_t)(key >> 44);
    res->err_layer = (uint32_t)(key >> 32) & 0xFFF;
    res->err_phase = (uint32_t)(key >> 24) & 0xFF;
    res->err_element = (uint32_t)key & 0xFFFFFF;
  }
  return rc;
}

/* Buffer offsets of the state, for the bindings: prompt, out, x, xb, q, o, y, h, logits,
 * scores, k, v, size (13 values). */
void orc_state_layout(const orc_model* m, uint32_t n_prompt, uint32_t max_tokens, uint64_t* out13) {
  uint32_t cfg[7];
  model_cfg(m, cfg);
  orc_layout L = layout_of(cfg, n_prompt, max_tokens);
  memcpy(out13, &L, sizeof(L));
}

/* ------------------------------------------------------------------ tokenizer
 * "The forward pass, in order", phases 0 to 2, and the text of a generated token
 * ("Sampling", last paragraph), over a vocabulary in llama2.c's tokenizer file layout:
 * u32 longest token length, then per token f32 score, i32 byte length, the bytes.
 * Readings: r24 ties between merges of equal score go to the leftmost pair; r25 every
 * adjacent pair is looked up, the opening token's included. */

typedef struct {
  uint32_t n, max_len;
  float* score;
  uint32_t* len;
  const uint8_t** str;
  uint32_t* sorted; /* token ids in byte-string order, for the binary search */
  uint8_t* blob;
} orc_vocab;

static int bytes_cmp(const uint8_t* a, uint32_t la, const uint8_t* b, uint32_t lb) {
  uint32_t m = la < lb ? la : lb;
  int c = memcmp(a, b, m);
  if (c) return c;
  return la < lb ? -1 : la > lb ? 1 : 0;
}

static const orc_vocab* g_sort_vocab;
static int sort_cmp(const void* x, const void* y) {
  uint32_t a = *(const uint32_t*)x, b = *(const uint32_t*)y;
  const orc_vocab* v = g_sort_vocab;
  return bytes_cmp(v->str[a], v->len[a], v->str[b], v->len[b]);
}

/* Opens a vocabulary of n tokens.  Returns 0, or 2 for a blob that does not hold them or
 * that repeats a string. */
int orc_vocab_open(const uint8_t* blob, uint64_t blob_len, uint32_t n, orc_vocab** out) {
  *out = NULL;
  if (blob_len < 4 || n == 0) return 2;
  orc_vocab* v = (orc_vocab*)calloc(1, sizeof(orc_vocab));
  v->n = n;
  v->blob = (uint8_t*)malloc(blob_len);
  memcpy(v->blob, blob, blob_len);
  v->score = (float*)malloc(4ull * n);
  v->len = (uint32_t*)malloc(4ull * n);
  v->str = (const uint8_t**)malloc(sizeof(uint8_t*) * n);
  v->sorted = (uint32_t*)malloc(4ull * n);
  uint64_t off = 4;
  for (uint32_t i = 0; i < n; ++i) {
    int32_t l;
    if (off + 8 > blob_len) goto bad;
    memcpy(&v->score[i], v->blob + off, 4);
    memcpy(&l, v->blob + off + 4, 4);
    off += 8;
    if (l < 0 || off + (uint64_t)l > blob_len) goto bad;
    v->len[i] = (uint32_t)l;
    if ((uint32_t)l > v->max_len) v->max_len = (uint32_t)l;
    v->str[i] = v->blob + off;
    off += (uint64_t)l;
    v->sorted[i] = i;
  }
  g_sort_vocab = v;
  qsort(v->sorted, n, 4, sort_cmp);
  for (uint32_t i = 1; i < n; ++i) /* repeated strings would make a lookup ambiguous */
    if (sort_cmp(&v->sorted[i - 1], &v->sorted[i]) == 0) goto bad;
  *out = v;
  return 0;
bad:
  free(v->blob); free(v->score); free(v->len); free(v->str); free(v->sorted); free(v);
  return 2;
}

void orc_vocab_close(orc_vocab* v) {
  if (!v) return;
  free(v->blob); free(v->score); free(v->len); free(v->str); free(v->sorted); free(v);
}

/* "A lookup is a binary search over the sorted token ids": the id of the token whose
 * bytes are s, or -1. */
int64_t orc_vocab_lookup(const orc_vocab* v, const uint8_t* s, uint32_t len) {
  uint32_t lo = 0, hi = v->n;
  while (lo < hi) {
    uint32_t mid = (lo + hi) / 2, t = v->sorted[mid];
    int c = bytes_cmp(v->str[t], v->len[t], s, len);
    if (c == 0) return t;
    if (c < 0) lo = mid + 1; else hi = mid;
  }
  return -1;
}

/* Byte length of the UTF-8 character starting at s (at most left bytes), 0 if not a valid
 * character (bad lead byte, truncated, bad continuation, overlong or surrogate). */
static uint32_t utf8_char(const uint8_t* s, uint32_t left) {
  uint8_t c = s[0];
  uint32_t n;
  uint32_t cp;
  if (c < 0x80) return 1;
  if ((c & 0xE0) == 0xC0) { n = 2; cp = c & 0x1F; }
  else if ((c & 0xF0) == 0xE0) { n = 3; cp = c & 0x0F; }
  else if ((c & 0xF8) == 0xF0) { n = 4; cp = c & 0x07; }
  else return 0;
  if (n > left) return 0;
  for (uint32_t i = 1; i < n; ++i) {
    if ((s[i] & 0xC0) != 0x80) return 0;
    cp = (cp << 6) | (s[i] & 0x3F);
  }
  if ((n == 2 && cp < 0x80) || (n == 3 && cp < 0x800) || (n == 4 && cp < 0x10000)) return 0;
  if (cp > 0x10FFFF || (cp >= 0xD800 && cp <= 0xDFFF)) return 0;
  return n;
}

/* Phases 0 to 2 on a prompt of len bytes: the opening token 1, the token of a single space
 * when the prompt has text, one token per character (or per byte, id byte + 3, for a
 * character with no token), then the merges.  Writes at most cap ids.  Returns 0, 6 for a
 * prompt over 1,024 bytes, with a zero byte or not UTF-8, or 4 when cap is too small. */
int orc_encode(const orc_vocab* v, const uint8_t* text, uint32_t len, uint32_t* ids, uint32_t cap,
               uint32_t* n_out) {
  *n_out = 0;
  if (len > 1024) return 6;
  for (uint32_t i = 0; i < len;) {
    if (text[i] == 0) return 6;
    uint32_t k = utf8_char(text + i, len - i);
    if (!k) return 6;
    i += k;
  }
  uint32_t* t = (uint32_t*)malloc(4ull * (len + 2));
  uint32_t n = 0;
  t[n++] = 1;                                                  /* phase 0 */
  if (len) {
    const uint8_t sp = ' ';
    int64_t id = orc_vocab_lookup(v, &sp, 1);
    t[n++] = id >= 0 ? (uint32_t)id : (uint32_t)sp + 3;
  }
  for (uint32_t i = 0; i < len;) {                             /* phase 1 */
    uint32_t k = utf8_char(text + i, len - i);
    int64_t id = orc_vocab_lookup(v, text + i, k);
    if (id >= 0) t[n++] = (uint32_t)id;
    else for (uint32_t b = 0; b < k; ++b) t[n++] = (uint32_t)text[i + b] + 3;
    i += k;
  }
  uint8_t* buf = (uint8_t*)malloc(2ull * v->max_len + 2);       /* phase 2 */
  for (;;) {
    float best = 0;
    int64_t best_id = -1;
    uint32_t best_i = 0;
    for (uint32_t i = 0; i + 1 < n; ++i) {
      uint32_t la = v->len[t[i]], lb = v->len[t[i + 1]];
      memcpy(buf, v->str[t[i]], la);
      memcpy(buf + la, v->str[t[i + 1]], lb);
      int64_t id = orc_vocab_lookup(v, buf, la + lb);
      if (id >= 0 && (best_id < 0 || v->score[id] > best)) {
        best = v->score[id];
        best_id = id;
        best_i = i;
      }
    }
    if (best_id < 0) break;
    t[best_i] = (uint32_t)best_id;
    memmove(t + best_i + 1, t + best_i + 2, 4ull * (n - best_i - 2));
    --n;
  }
  free(buf);
  int rc = 0;
  if (n > cap) rc = 4;
  else memcpy(ids, t, 4ull * n);
  *n_out = n;
  free(t);
  return rc;
}

/* The text of token tok generated after token prev ("Sampling"): the token's bytes, a
 * leading space dropped right after the opening token, <0xXX> as that one byte, nothing
 * for tokens 1 and 2.  Writes at most cap bytes; returns the byte count. */
uint32_t orc_decode_piece(const orc_vocab* v, uint32_t prev, uint32_t tok, uint8_t* out, uint32_t cap) {
  if (tok >= v->n || tok == 1 || tok == 2) return 0;
  const uint8_t* s = v->str[tok];
  uint32_t l = v->len[tok];
  if (prev == 1 && l && s[0] == ' ') { ++s; --l; }
  if (l == 6 && s[0] == '<' && s[1] == '0' && s[2] == 'x' && s[5] == '>') {
    unsigned val = 0;
    int ok = 1;
    for (int i = 3; i < 5; ++i) {
      uint8_t c = s[i];
      unsigned d = c >= '0' && c <= '9' ? c - '0' : c >= 'A' && c <= 'F' ? c - 'A' + 10 :
                   c >= 'a' && c <= 'f' ? c - 'a' + 10 : 16;
      if (d == 16) ok = 0;
      val = val * 16 + d;
    }
    if (ok) {
      if (cap) out[0] = (uint8_t)val;
      return 1;
    }
  }
  uint32_t w = l < cap ? l : cap;
  memcpy(out, s, w);
  return w;
}

/* ------------------------------------------------------------------ the page's state
 * "The resumable state": the CURTAST2 state (a 128-byte header and text-mode buffers) and
 * the phases of "The forward pass, in order" run one step at a time, a step being one
 * phase of one layer of one position (phase 9 one head a step, the row field naming the
 * head), so that a turn can stop at any phase boundary, mid-layer included, and another
 * target can go on from the bytes.  Readings: r27 the working vectors between phases
 * (activations x; w0 the normalised vector, then the output rows before their residual;
 * w1 the queries; w2 the heads' outputs; gate and up, then SiLU's output in gate); r28 the
 * tokenizer phases 0 to 2 are one step; r29 a step is all or nothing: a store that does
 * not fit leaves the state as it was before the step and the turn returns 8. */

enum { P_PHASE = 8, P_LAYER = 12, P_ROW = 16, P_POS = 20, P_TOKEN = 24, P_PBYTES = 28, P_NPTOK = 32,
       P_MAXTOK = 36, P_TEMP = 40, P_GEN = 44, P_TEXTLEN = 48, P_SEED = 72, P_TURNS = 80,
       P_MAXSCORE = 88, P_CHOSEN = 96, P_SPASS = 100, P_SUM = 104, P_DRAW = 112, P_ASTAGE = 120,
       P_AINDEX = 124 };

typedef struct {
  uint64_t prompt, ptok, out, text, x, w0, w1, w2, gate, up, logits, scores, k, v, size;
  uint32_t cache;
} orc_page_layout;

static orc_page_layout page_layout(const orc_model* m, uint32_t prompt_bytes, uint32_t max_tokens) {
  orc_page_layout L;
  uint64_t cache = (uint64_t)prompt_bytes + max_tokens + 1;
  if (cache > m->context) cache = m->context;
  uint64_t n = 128;
  L.prompt = n; n = up8(n + prompt_bytes);
  L.ptok = n; n = up8(n + 4ull * (prompt_bytes + 2));
  L.out = n; n = up8(n + 4ull * max_tokens);
  L.text = n; n = up8(n + 128ull * max_tokens);
  L.x = n; L.w0 = n + 8ull * m->dim; L.w1 = n + 16ull * m->dim; L.w2 = n + 24ull * m->dim;
  n = up8(n + 32ull * m->dim);
  L.gate = n; L.up = n + 8ull * m->hidden; n = up8(n + 16ull * m->hidden);
  L.logits = n; n = up8(n + 8ull * m->vocab);
  L.scores = n; n = up8(n + 8 * cache);
  L.k = n; n = up8(n + 4ull * m->layers * cache * m->kv_dim);
  L.v = n; n = up8(n + 4ull * m->layers * cache * m->kv_dim);
  L.size = n;
  L.cache = (uint32_t)cache;
  return L;
}

uint64_t orc_page_size(const orc_model* m, uint32_t prompt_bytes, uint32_t max_tokens) {
  return page_layout(m, prompt_bytes, max_tokens).size;
}

/* Buffer offsets, for the bindings: prompt, ptok, out, text, x, w0, w1, w2, gate, up,
 * logits, scores, k, v, size (15 values) and the cache positions. */
void orc_page_layout_of(const orc_model* m, uint32_t prompt_bytes, uint32_t max_tokens, uint64_t* out16) {
  orc_page_layout L = page_layout(m, prompt_bytes, max_tokens);
  memcpy(out16, &L, 15 * 8);
  out16[15] = L.cache;
}

/* "The Rust API", init_state: a fresh header and the prompt.  Errors: 4 wrong length, 6
 * max tokens 0 or above the context, a temperature above 16, a prompt over 1,024 bytes. */
int orc_page_init(const orc_model* m, uint8_t* st, uint64_t len, const uint8_t* prompt, uint32_t plen,
                  uint32_t max_tokens, uint32_t temperature_q16, uint64_t seed) {
  if (max_tokens == 0 || max_tokens > m->context || temperature_q16 > (16u << 16) || plen > 1024) return 6;
  orc_page_layout L = page_layout(m, plen, max_tokens);
  if (len != L.size) return 4;
  memset(st, 0, len);
  memcpy(st, "CURTAST2", 8);
  wr32(st + P_PBYTES, plen);
  wr32(st + P_MAXTOK, max_tokens);
  wr32(st + P_TEMP, temperature_q16);
  wr64(st + P_SEED, seed ? seed : 0x9E3779B97F4A7C15ull);
  memcpy(st + L.prompt, prompt, plen);
  return 0;
}

static int store_fit(int32_t* dst, const int64_t* src, uint32_t n) {
  for (uint32_t j = 0; j < n; ++j)
    if (!orc_fits32(src[j])) return (int)j;
  for (uint32_t j = 0; j < n; ++j) dst[j] = (int32_t)src[j];
  return -1;
}

/* One step from the state's cursor.  Returns 0, or an error (3 finished or foreign state,
 * 6 bad prompt, 7 context exceeded, 8 a store that does not fit: nothing changed). */
static int page_step(const orc_model* m, const orc_vocab* voc, uint8_t* st, const orc_page_layout* L) {
  const uint32_t phase = rd32(st + P_PHASE), l = rd32(st + P_LAYER), pos = rd32(st + P_POS);
  const uint32_t d = m->dim, hd = m->head_dim, kvd = m->kv_dim, hid = m->hidden, cache = L->cache;
  const uint32_t np = rd32(st + P_NPTOK);
  int64_t *x = (int64_t*)(st + L->x), *w0 = (int64_t*)(st + L->w0), *w1 = (int64_t*)(st + L->w1);
  int64_t *w2 = (int64_t*)(st + L->w2), *g = (int64_t*)(st + L->gate), *u = (int64_t*)(st + L->up);
  int64_t* logits = (int64_t*)(st + L->logits);
  int32_t *K = (int32_t*)(st + L->k), *V = (int32_t*)(st + L->v);
  uint32_t* ptok = (uint32_t*)(st + L->ptok);
  uint32_t* out = (uint32_t*)(st + L->out);
  const orc_layer* W = l < m->layers ? &m->layer[l] : NULL;
  int32_t* Kp = K + ((uint64_t)l * cache + pos) * kvd; /* the page's order: [layer][position][kv] */
  int32_t* Vp = V + ((uint64_t)l * cache + pos) * kvd;
  switch (phase) {
    case 0: { /* phases 0 to 2: the prompt's tokens */
      uint32_t n = 0, plen = rd32(st + P_PBYTES);
      int rc = orc_encode(voc, st + L->prompt, plen, ptok, plen + 2, &n);
      if (rc) return rc;
      if ((uint64_t)n + rd32(st + P_MAXTOK) > cache) return 7;
      wr32(st + P_NPTOK, n);
      wr32(st + P_POS, 0);
      wr32(st + P_TOKEN, ptok[0]);
      wr32(st + P_PHASE, 3);
      return 0;
    }
    case 3: {
      uint32_t tok = rd32(st + P_TOKEN);
      if (tok >= m->vocab) return 3;
      orc_embed(m->embed + (uint64_t)tok * d, m->embed_scale[tok], d, x);
      wr32(st + P_LAYER, 0);
      wr32(st + P_PHASE, 4);
      return 0;
    }
    case 4: orc_rmsnorm(x, W->attn_norm, d, w0); break;
    case 5: orc_matrow(W->wq, d, W->sq, d, d, w0, w1); break;
    case 6: case 7: {
      int64_t* tmp = (int64_t*)malloc(8ull * kvd);
      orc_matrow(phase == 6 ? W->wk : W->wv, d, phase == 6 ? W->sk : W->sv, kvd, d, w0, tmp);
      int bad = store_fit(phase == 6 ? Kp : Vp, tmp, kvd);
      free(tmp);
      if (bad >= 0) return 8;
      break;
    }
    case 8: {
      const int32_t* rope = m->rope + (uint64_t)pos * hd;
      int32_t* kk = (int32_t*)malloc(4ull * kvd);
      for (uint32_t i = 0; i < kvd; i += 2) {
        uint32_t j = (i % hd) / 2;
        int64_t a2, b2;
        orc_rotate(Kp[i], Kp[i + 1], rope[2 * j], rope[2 * j + 1], &a2, &b2);
        if (!orc_fits32(a2) || !orc_fits32(b2)) { free(kk); return 8; }
        kk[i] = (int32_t)a2;
        kk[i + 1] = (int32_t)b2;
      }
      memcpy(Kp, kk, 4ull * kvd);
      free(kk);
      for (uint32_t i = 0; i < d; i += 2) {
        uint32_t j = (i % hd) / 2;
        orc_rotate(w1[i], w1[i + 1], rope[2 * j], rope[2 * j + 1], &w1[i], &w1[i + 1]);
      }
      wr32(st + P_ROW, 0);
      wr32(st + P_ASTAGE, 0);
      wr32(st + P_AINDEX, 0);
      break;
    }
    case 9: { /* one head a step */
      uint32_t h = rd32(st + P_ROW);
      uint32_t kvh = h / (m->heads / m->kv_heads);
      const int32_t* K0 = K + (uint64_t)l * cache * kvd + (uint64_t)kvh * hd;
      const int32_t* V0 = V + (uint64_t)l * cache * kvd + (uint64_t)kvh * hd;
      orc_attention_head(w1 + (uint64_t)h * hd, K0, V0, kvd, pos + 1, hd, m->inv_sqrt, m->exp_tab,
                         (int64_t*)(st + L->scores), w2 + (uint64_t)h * hd);
      if (h + 1 < m->heads) {
        wr32(st + P_ROW, h + 1);
        return 0;
      }
      wr32(st + P_ROW, 0);
      break;
    }
    case 10: orc_matrow(W->wo, d, W->so, d, d, w2, w0); break;
    case 11: residual(x, w0, d); orc_rmsnorm(x, W->ffn_norm, d, w0); break;
    case 12: orc_matrow(W->w1, d, W->s1, hid, d, w0, g); break;
    case 13: orc_matrow(W->w3, d, W->s3, hid, d, w0, u); break;
    case 14: orc_silu_gate(g, u, hid, m->silu_tab, g); break;
    case 15: orc_matrow(W->w2, hid, W->s2, d, hid, g, w0); break;
    case 16: {
      residual(x, w0, d);
      if (l + 1 < m->layers) {
        wr32(st + P_LAYER, l + 1);
        wr32(st + P_PHASE, 4);
      } else if (pos + 1 < np) {                          /* the next prompt position */
        wr32(st + P_POS, pos + 1);
        wr32(st + P_TOKEN, ptok[pos + 1]);
        wr32(st + P_LAYER, 0);
        wr32(st + P_PHASE, 3);
      } else {
        wr32(st + P_PHASE, 17);
      }
      return 0;
    }
    case 17: orc_rmsnorm(x, m->final_norm, d, w0); break;
    case 18: orc_matrow(m->cls, d, m->cls_scale, m->vocab, d, w0, logits); break;
    case 19: {
      uint64_t state = rd64(st + P_SEED), z, draw;
      int64_t mx;
      uint32_t t = orc_sample(logits, m->vocab, rd32(st + P_TEMP), m->exp_tab, &state, &mx, &z, &draw);
      uint32_t gen = rd32(st + P_GEN), tl = rd32(st + P_TEXTLEN);
      uint32_t prev = pos < np ? ptok[pos] : out[gen - 1];
      out[gen] = t;
      tl += orc_decode_piece(voc, prev, t, st + L->text + tl, 128);
      wr32(st + P_GEN, gen + 1);
      wr32(st + P_TEXTLEN, tl);
      wr64(st + P_SEED, state);
      wr64(st + P_MAXSCORE, (uint64_t)mx);
      wr32(st + P_CHOSEN, t);
      wr64(st + P_SUM, z);
      wr64(st + P_DRAW, draw);
      if (t == 1 || t == 2 || gen + 1 == rd32(st + P_MAXTOK)) {
        wr32(st + P_PHASE, 20);
      } else {
        wr32(st + P_POS, pos + 1);
        wr32(st + P_TOKEN, t);
        wr32(st + P_LAYER, 0);
        wr32(st + P_PHASE, 3);
      }
      return 0;
    }
    default: return 3;
  }
  wr32(st + P_PHASE, phase + 1);
  return 0;
}

/* "The Rust API", turn, at step granularity: up to n_steps steps.  Returns 0 or the error
 * of the step that failed (that step changed nothing); *steps receives the steps run. */
int orc_page_turn(const orc_model* m, const orc_vocab* voc, uint8_t* st, uint64_t len, uint32_t n_steps,
                  uint32_t* steps) {
  *steps = 0;
  if (len < 128 || memcmp(st, "CURTAST2", 8) != 0) return 3;
  orc_page_layout L = page_layout(m, rd32(st + P_PBYTES), rd32(st + P_MAXTOK));
  if (len != L.size) return 3;
  int rc = 0;
  for (uint32_t i = 0; i < n_steps && rd32(st + P_PHASE) != 20; ++i) {
    rc = page_step(m, voc, st, &L);
    if (rc) break;
    ++*steps;
  }
  wr64(st + P_TURNS, rd64(st + P_TURNS) + 1);
  return rc;
}
