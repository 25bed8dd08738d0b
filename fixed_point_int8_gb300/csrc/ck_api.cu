// libck host API: artifact loading into HBM, state set-up and the phase sequencer that
// replays one position's kernels as a CUDA graph ("The inference core": "The forward pass,
// in order", "The resumable state", "The Rust API", "Core errors").
#include <algorithm>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <new>
#include <thread>
#include <vector>

#include "ck_internal.cuh"

using namespace ck;

struct ck_model {
  ck_config cfg;
  uint32_t head_dim, kv_dim, inv_sqrt, flags, pitch_d, pitch_h;
  int device, num_sms;
  uint8_t* dev;
  size_t dev_len;
  const uint8_t* embed;
  const uint32_t* embed_scale;
  const uint8_t* cls;
  const uint32_t* cls_scale;
  const int32_t* final_norm;
  const int32_t* rope;
  const uint32_t* exp_tab;
  const int32_t* silu_tab;
  uint32_t* scratch;  // small device scratch inside dev (ck_argmax result)
  DevLayer* dev_layers;  // the layer table in device memory (read by the one-position kernel)
  int path;              // CK_PATH_*
  uint32_t max_slots;    // cap on the one-position kernel's ring slots (0: as many as fit)
  uint32_t att_full;     // positions every block of a head scores itself (0: default)
  uint32_t pf_kb;        // L2 prefetch distance of the one-position kernel, KB per block
  uint32_t sync_polls;   // polls of the one-position kernel's barriers (0: the default)
                         // (0: default)
  int smem_optin;        // largest shared memory a block may opt into
  size_t step_smem;      // dynamic shared memory available to the one-position kernel
  std::vector<DevLayer> layers;
  uint32_t pf_cap;       // prompt positions per layer-major chunk (0: position by position)
  uint8_t* pf_work;      // device scratch of the batched kernels, allocated at first use
  size_t pf_bytes;
  uint32_t pf_wcap;      // rows the scratch is laid out for
  bool pf_configured;
  cudaStream_t capture;
  struct Graph {
    void* state;
    size_t len;
    bool generating;
    int path;
    cudaGraphExec_t exec;
  };
  std::vector<Graph> graphs;
  struct BatchGraph {  // a batched pass's kernels for a row count and position bound
    uint32_t n, max_positions;
    uint8_t* work;
    uint32_t cap;
    cudaGraphExec_t exec;
  };
  std::vector<BatchGraph> bgraphs;
};

namespace {

constexpr uint32_t kTable = 4097;
constexpr uint32_t kDefaultPrefillChunk = 256;  // prompt positions per layer-major chunk
constexpr uint32_t kMaxPrefillChunk = 4096;

uint32_t rd32(const uint8_t* p) { uint32_t v; memcpy(&v, p, 4); return v; }
uint64_t rd64(const uint8_t* p) { uint64_t v; memcpy(&v, p, 8); return v; }

int check_config(const ck_config& c) {
  if (!c.dim || !c.hidden || !c.layers || !c.heads || !c.kv_heads || !c.vocab || !c.context)
    return CK_INVALID_CONFIG;
  if (c.dim % c.heads || c.heads % c.kv_heads) return CK_INVALID_CONFIG;
  const uint32_t hd = c.dim / c.heads;
  if (hd < 4 || hd > 128 || (hd & (hd - 1))) return CK_INVALID_CONFIG;
  if (c.dim > 16384 || c.hidden > 16384 || c.layers > 4095 || c.vocab > (1u << 20) ||
      c.context > 32768)
    return CK_INVALID_CONFIG;
  return CK_OK;
}

struct Parsed {
  ck_config cfg;
  uint32_t inv_sqrt, flags;
  std::vector<const uint8_t*> t;
};

int parse_artifact(const void* artifact, size_t len, Parsed* out) {
  if (!artifact || !out) return CK_INVALID_ARGUMENT;
  const uint8_t* a = static_cast<const uint8_t*>(artifact);
  if (len < 64 || memcmp(a, "CKMODEL1", 8) != 0) return CK_INVALID_FORMAT;
  ck_config c;
  memcpy(&c, a + 8, sizeof(c));
  int rc = check_config(c);
  if (rc) return rc;
  const uint32_t n = rd32(a + 44);
  if (n != 8 + 16 * c.layers || rd64(a + 48) != len || 64 + 16ull * n > len) return CK_INVALID_FORMAT;
  const uint64_t d = c.dim, h = c.hidden, v = c.vocab, kv = (uint64_t)c.dim / c.heads * c.kv_heads;
  const bool tied = rd32(a + 40) & 1u;
  const uint64_t glob[8] = {v * d, 4 * v, 4 * d, tied ? 0 : v * d, tied ? 0 : 4 * v,
                            4ull * c.context * (c.dim / c.heads), 4ull * kTable, 4ull * kTable};
  const uint64_t lay[16] = {4 * d, d * d, 4 * d, kv * d, 4 * kv, kv * d, 4 * kv, d * d,
                            4 * d, 4 * d, h * d, 4 * h, h * d, 4 * h, d * h, 4 * d};
  out->t.assign(n, nullptr);
  for (uint32_t i = 0; i < n; ++i) {
    const uint64_t off = rd64(a + 64 + 16ull * i), tl = rd64(a + 64 + 16ull * i + 8);
    const uint64_t want = i < 8 ? glob[i] : lay[(i - 8) % 16];
    if (tl != want) return CK_INVALID_FORMAT;
    if (tl && (off > len || tl > len - off || off % 4)) return CK_INVALID_FORMAT;
    out->t[i] = a + off;
  }
  out->cfg = c;
  out->inv_sqrt = rd32(a + 36);
  out->flags = rd32(a + 40);
  return CK_OK;
}

// Offsets of the device model layout.
struct DevPlan {
  uint64_t embed, embed_scale, cls, cls_scale, final_norm, rope, exp_tab, silu_tab, scratch, table;
  struct L { uint64_t wqkv, sqkv, wo, so, w13, s13, w2, s2, an, fn; };
  std::vector<L> layers;
  uint64_t total;
};

DevPlan plan_device(const ck_config& c, bool tied) {
  DevPlan P;
  const uint64_t pd = pad128(c.dim), ph = pad128(c.hidden), hd = c.dim / c.heads;
  const uint64_t kv = hd * c.kv_heads;
  uint64_t off = 0;
  auto take = [&](uint64_t bytes) { uint64_t o = off; off = align256(off + bytes); return o; };
  P.embed = take(c.vocab * pd);
  P.embed_scale = take(4ull * c.vocab);
  P.cls = tied ? P.embed : take(c.vocab * pd);
  P.cls_scale = tied ? P.embed_scale : take(4ull * c.vocab);
  P.final_norm = take(4ull * c.dim);
  P.rope = take(4ull * c.context * hd);
  P.exp_tab = take(4ull * kTable);
  P.silu_tab = take(4ull * kTable);
  P.layers.resize(c.layers);
  for (uint32_t l = 0; l < c.layers; ++l) {
    DevPlan::L& L = P.layers[l];
    L.wqkv = take((c.dim + 2 * kv) * pd);
    L.sqkv = take(4 * (c.dim + 2 * kv));
    L.wo = take(c.dim * pd);
    L.so = take(4ull * c.dim);
    L.w13 = take(2ull * c.hidden * pd);
    L.s13 = take(8ull * c.hidden);
    L.w2 = take(c.dim * ph);
    L.s2 = take(4ull * c.dim);
    L.an = take(4ull * c.dim);
    L.fn = take(4ull * c.dim);
  }
  P.scratch = take(256);
  P.table = take(sizeof(DevLayer) * (uint64_t)c.layers);
  P.total = off;
  return P;
}

#define CK_CUDA(call)                          \
  do {                                         \
    cudaError_t e_ = (call);                   \
    if (e_ != cudaSuccess) return CK_CUDA_ERROR; \
  } while (0)

inline cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }

// Uploads a matrix of `rows` rows of `cols` bytes (row r at row_ptr(r)) to dst in
// column-group layout with `pitch` columns (a multiple of 128; padding bytes zero).  The
// host reorders into `stage` with a few threads, then one copy; a copy from pageable
// memory returns once the bytes are staged, so the buffer may be reused right after.
template <typename RowFn>
cudaError_t upload_grouped(uint8_t* dst, uint32_t rows, uint32_t cols, uint32_t pitch, RowFn row_ptr,
                           std::vector<uint8_t>& stage, cudaStream_t s) {
  if (!rows) return cudaSuccess;
  const size_t bytes = (size_t)rows * pitch;
  if (stage.size() < bytes) stage.resize(bytes);
  uint8_t* out = stage.data();
  const uint32_t groups = pitch / kGroupCols;
  auto work = [&](uint32_t r0, uint32_t r1) {
    for (uint32_t r = r0; r < r1; ++r) {
      const uint8_t* src = row_ptr(r);
      for (uint32_t g = 0; g < groups; ++g) {
        uint8_t* d = out + ((size_t)g * rows + r) * kGroupCols;
        for (uint32_t j = 0; j < 8; ++j) {
          const uint32_t col = g * kGroupCols + 16 * j;
          uint8_t* chunk = d + ((j ^ (r & 7u)) << 4);
          const uint32_t n = col >= cols ? 0u : (cols - col < 16 ? cols - col : 16u);
          if (n) memcpy(chunk, src + col, n);
          if (n < 16) memset(chunk + n, 0, 16 - n);
        }
      }
    }
  };
  unsigned nt = std::thread::hardware_concurrency();
  if (nt < 1) nt = 1;
  if (nt > 16) nt = 16;
  if ((size_t)rows * pitch < (1u << 22) || rows < nt) nt = 1;
  if (nt == 1) {
    work(0, rows);
  } else {
    std::vector<std::thread> th;
    for (unsigned t = 0; t < nt; ++t)
      th.emplace_back(work, (uint32_t)((uint64_t)rows * t / nt), (uint32_t)((uint64_t)rows * (t + 1) / nt));
    for (auto& t : th) t.join();
  }
  return cudaMemcpyAsync(dst, out, bytes, cudaMemcpyHostToDevice, s);
}

// ------------------------------------------------------------------ small kernels

// Phase 3: x[i] = ((byte - 128) * scale) >> 8 over the row of this position's token.
// It also clears the position's sums of squares (nslots words at `slots`), which the
// kernels producing each residual add into.
__global__ void k_embed(uint8_t* st, uint64_t off_prompt, uint64_t off_out, int64_t* x,
                        const uint8_t* embed, const uint32_t* scale, uint32_t pitch, uint32_t dim,
                        uint32_t vocab, unsigned long long* slots, uint32_t nslots) {
  if (hdr_ld<uint32_t>(st, kHPhase) != CK_PHASE_RUNNING) return;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < nslots; i += gridDim.x * blockDim.x) slots[i] = 0;
  const uint32_t pos = hdr_ld<uint32_t>(st, kHPosition), np = hdr_ld<uint32_t>(st, kHNPrompt);
  const uint32_t tok = pos < np ? reinterpret_cast<const uint32_t*>(st + off_prompt)[pos]
                                : reinterpret_cast<const uint32_t*>(st + off_out)[pos - np];
  if (tok >= vocab) {  // a state edited outside the library: stop instead of reading past the table
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      hdr<uint32_t>(st, kHError) = CK_INVALID_STATE;
      hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
    }
    return;
  }
  (void)pitch;
  const int64_t s = (int64_t)__ldg(scale + tok);
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < dim; i += gridDim.x * blockDim.x)
    x[i] = ((int64_t)embed[grouped_offset(vocab, tok, i)] - 128) * s >> 8;
}

// End of a prompt position (its last residual is already in x): the cursor moves on, or the
// state is marked failed if a cache store did not fit.
__global__ void k_finish_prompt(uint8_t* st) {
  if (hdr_ld<uint32_t>(st, kHPhase) != CK_PHASE_RUNNING) return;
  if (threadIdx.x == 0) {
    if (hdr_ld<uint64_t>(st, kHErrKey) != kNoError) {
      hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
      hdr<uint32_t>(st, kHError) = CK_ARITHMETIC;
    } else {
      hdr<uint32_t>(st, kHPosition) += 1;
    }
  }
}

constexpr int kArgThreads = 1024;

// First index of the largest logit (strictly greater wins while scanning upward).
__device__ void block_argmax(const int64_t* l, uint32_t n, long long* best_v, uint32_t* best_i) {
  __shared__ long long sv[kArgThreads / 32];
  __shared__ uint32_t si[kArgThreads / 32];
  long long bv = LLONG_MIN;
  uint32_t bi = 0xFFFFFFFFu;
  // eight loads a thread in flight, then compared in index order (the first of equal
  // maxima stays)
  constexpr int kU = 8;
  for (uint32_t i0 = threadIdx.x; i0 < n; i0 += kU * blockDim.x) {
    long long v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const uint32_t i = i0 + u * blockDim.x;
      v[u] = i < n ? l[i] : LLONG_MIN;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const uint32_t i = i0 + u * blockDim.x;
      if (i < n && (bi == 0xFFFFFFFFu || v[u] > bv)) {
        bv = v[u];
        bi = i;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const long long ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const uint32_t oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (oi != 0xFFFFFFFFu && (bi == 0xFFFFFFFFu || ov > bv || (ov == bv && oi < bi))) {
      bv = ov;
      bi = oi;
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x / 32); ++w) {
      if (si[w] != 0xFFFFFFFFu && (bi == 0xFFFFFFFFu || sv[w] > bv || (sv[w] == bv && si[w] < bi))) {
        bv = sv[w];
        bi = si[w];
      }
    }
    *best_v = bv;
    *best_i = bi;
  }
}

// Phase 19 ("Sampling": the maximum pass, and above temperature zero the sum and draw
// passes) plus the end of a generating position.
__global__ void __launch_bounds__(kArgThreads) k_sample_finish(uint8_t* st, uint64_t off_out,
                                                              const int64_t* logits, uint32_t vocab,
                                                              const uint32_t* exp_tab) {
  __shared__ unsigned long long gsum[kSampleGroups];
  __shared__ long long max_v;
  __shared__ uint32_t max_i;
  if (hdr_ld<uint32_t>(st, kHPhase) != CK_PHASE_RUNNING) return;
  if (hdr_ld<uint64_t>(st, kHErrKey) != kNoError) {
    if (threadIdx.x == 0) {
      hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
      hdr<uint32_t>(st, kHError) = CK_ARITHMETIC;
    }
    return;
  }
  long long bv;
  uint32_t bi;
  block_argmax(logits, vocab, &bv, &bi);
  if (threadIdx.x == 0) {
    max_v = bv;
    max_i = bi;
  }
  __syncthreads();
  bv = max_v;
  bi = max_i;
  const uint32_t temp = hdr_ld<uint32_t>(st, kHTemp);
  unsigned long long state = hdr_ld<unsigned long long>(st, kHSeed), z = 0, draw = 0;
  if (temp != 0) {
    const SampleOut so = block_sample(reinterpret_cast<const long long*>(logits), vocab, bv, temp,
                                      exp_tab, state, gsum, kArgThreads / 32,
                                      [] { __syncthreads(); });
    bi = so.token;
    state = so.state;
    z = so.sum;
    draw = so.draw;
  }
  if (threadIdx.x == 0) {
    const uint32_t gen = hdr_ld<uint32_t>(st, kHGenerated);
    if (gen >= hdr_ld<uint32_t>(st, kHMaxTok)) {  // unreachable for states the turn validated
      hdr<uint32_t>(st, kHError) = CK_INVALID_STATE;
      hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
      return;
    }
    reinterpret_cast<uint32_t*>(st + off_out)[gen] = bi;
    hdr<uint32_t>(st, kHGenerated) = gen + 1;
    hdr<uint32_t>(st, kHLastTok) = bi;
    hdr<long long>(st, kHMaxLogit) = bv;
    hdr<unsigned long long>(st, kHSeed) = state;
    hdr<unsigned long long>(st, kHExpSum) = z;
    hdr<unsigned long long>(st, kHDraw) = draw;
    const bool stop = (hdr_ld<uint32_t>(st, kHFlags) & CK_FLAG_STOP_TOKENS) && (bi == 1 || bi == 2);
    if (gen + 1 == hdr_ld<uint32_t>(st, kHMaxTok) || stop) hdr<uint32_t>(st, kHPhase) = CK_PHASE_DONE;
    hdr<uint32_t>(st, kHPosition) += 1;
  }
}

__global__ void __launch_bounds__(kArgThreads) k_argmax(const int64_t* logits, uint32_t vocab,
                                                       uint32_t* out) {
  long long bv;
  uint32_t bi;
  block_argmax(logits, vocab, &bv, &bi);
  if (threadIdx.x == 0) *out = bi;
}

// ------------------------------------------------------------------ state checks

struct HostHeader {
  uint8_t b[kHeaderBytes];
  uint32_t u32(uint32_t off) const { return rd32(b + off); }
  uint64_t u64(uint32_t off) const { return rd64(b + off); }
};

int read_header(const void* dev_state, HostHeader* h, cudaStream_t s) {
  CK_CUDA(cudaMemcpyAsync(h->b, dev_state, kHeaderBytes, cudaMemcpyDeviceToHost, s));
  CK_CUDA(cudaStreamSynchronize(s));
  return CK_OK;
}

// Checks that a state belongs to the model and has a valid cursor ("InvalidState").
int check_state(const ck_model* m, const void* dev_state, size_t len, const HostHeader& h,
                StateLayout* lay) {
  if (memcmp(h.b, "CKSTATE1", 8) != 0) return CK_INVALID_STATE;
  for (int i = 0; i < 7; ++i)
    if (h.u32(kHConfig + 4 * i) != (&m->cfg.dim)[i]) return CK_INVALID_STATE;
  const uint32_t np = h.u32(kHNPrompt), mt = h.u32(kHMaxTok);
  if (!np || !mt || mt > m->cfg.context || (uint64_t)np + mt - 1 > m->cfg.context) return CK_INVALID_STATE;
  *lay = state_layout(m->cfg, np, mt);
  if (len != lay->size || h.u32(kHCache) != lay->cache) return CK_INVALID_STATE;
  const uint32_t pos = h.u32(kHPosition);
  if (pos > lay->cache) return CK_INVALID_STATE;
  // tokens generated so far = generating positions already run
  const uint32_t gen = pos + 1 > np ? pos + 1 - np : 0;
  if (h.u32(kHGenerated) != gen) return CK_INVALID_STATE;
  (void)dev_state;
  return CK_OK;
}

int attention_cluster(uint32_t cache) {
  uint32_t c = (cache + 15) / 16;
  if (c < 1) c = 1;
  if (c > 8) c = 8;
  return (int)c;
}

// Enqueues one position's kernels (phases 3 to 16 for every layer, then 17 to 19 when the
// position generates a token).
int enqueue_position(const ck_model* m, uint8_t* st, const StateLayout& lay, bool generating,
                     cudaStream_t s) {
  const ck_config& c = m->cfg;
  int64_t* x = reinterpret_cast<int64_t*>(st + lay.x);
  int64_t* xb = reinterpret_cast<int64_t*>(st + lay.xb);
  int64_t* q = reinterpret_cast<int64_t*>(st + lay.q);
  int64_t* o = reinterpret_cast<int64_t*>(st + lay.o);
  int64_t* y = reinterpret_cast<int64_t*>(st + lay.y);
  int64_t* hbuf = reinterpret_cast<int64_t*>(st + lay.h);
  int64_t* logits = reinterpret_cast<int64_t*>(st + lay.logits);
  int32_t* K = reinterpret_cast<int32_t*>(st + lay.k);
  int32_t* V = reinterpret_cast<int32_t*>(st + lay.v);
  const size_t layer_words = (size_t)lay.cache * m->kv_dim;
  const int cl = attention_cluster(lay.cache);

  // sums of squares of the residuals: slot 2l feeds layer l's attention norm (l >= 1),
  // 2l + 1 its feed-forward norm, 2 layers the final norm; each is added up by the kernel that
  // produces the residual (O and DOWN epilogues) and read whole by the normalizing kernel
  unsigned long long* ss = reinterpret_cast<unsigned long long*>(st + lay.scores);
  const uint32_t nslots = 2 * c.layers + 1;
  // after them (256-byte aligned), where the work region holds it: the attention outputs'
  // sums before their >> 24, added into by every attention CTA, read by the O kernel and
  // cleared by the gate/up kernel for the next layer
  const uint32_t oacc_word = (nslots + 31) & ~31u;
  const bool use_oacc = 8ull * ((uint64_t)oacc_word + c.dim) <= lay.k - lay.scores;
  unsigned long long* oacc = use_oacc ? ss + oacc_word : nullptr;
  // after them, where the region holds it: the SiLU outputs as byte planes with the gate/up
  // CTAs' partial sums and ORs, written by the gate/up epilogue for the down kernel's prologue
  const uint32_t gu_grid = std::min<uint32_t>(c.hidden, (uint32_t)m->num_sms);
  const uint64_t off_hplanes = align256(8ull * ((uint64_t)oacc_word + c.dim));
  const uint64_t off_hparts = align256(off_hplanes + 8ull * m->pitch_h);
  const bool use_hplanes = use_oacc && off_hparts + 16ull * gu_grid <= lay.k - lay.scores;
  uint8_t* hplanes = use_hplanes ? st + lay.scores + off_hplanes : nullptr;
  unsigned long long* hparts =
      use_hplanes ? reinterpret_cast<unsigned long long*>(st + lay.scores + off_hparts) : nullptr;
  k_embed<<<(c.dim + 255) / 256, 256, 0, s>>>(st, lay.prompt, lay.out, x, m->embed, m->embed_scale,
                                              m->pitch_d, c.dim, c.vocab, ss,
                                              use_oacc ? oacc_word + c.dim : nslots);
  CK_CUDA(cudaGetLastError());
  int64_t* cur = x;  // the buffer holding the activations (x and xb take turns)
  for (uint32_t l = 0; l < c.layers; ++l) {
    const DevLayer& W = m->layers[l];
    // phases 4-8: attention norm, Q/K/V, cache stores, rotary
    MatrowParams p = {};
    p.W = W.wqkv;
    p.scale = W.sqkv;
    p.grouped = 1;
    p.pitch = m->pitch_d;
    p.rows = c.dim + 2 * m->kv_dim;
    p.cols = c.dim;
    p.pro = kProNorm;
    p.in = cur;
    p.norm_w = W.attn_norm;
    if (l > 0) p.ss_in = ss + 2 * l;  // layer 0's embedding: the prologue adds its squares up
    p.epi = kEpiQKV;
    p.out = q;
    p.q_rows = c.dim;
    p.kv_dim = m->kv_dim;
    p.head_dim = m->head_dim;
    p.layer = l;
    p.cache = lay.cache;
    p.kcache = K + l * layer_words;
    p.vcache = V + l * layer_words;
    p.rope = m->rope;
    p.state = st;
    CK_CUDA(launch_matrow(p, s, m->num_sms));
    // phase 9
    AttnParams a = {};
    a.state = st;
    a.q = q;
    a.o = o;
    a.kcache = K + l * layer_words;
    a.vcache = V + l * layer_words;
    a.exp_tab = m->exp_tab;
    a.heads = c.heads;
    a.kv_heads = c.kv_heads;
    a.head_dim = m->head_dim;
    a.kv_dim = m->kv_dim;
    a.inv_sqrt = m->inv_sqrt;
    a.cache = lay.cache;
    a.chunk_cap = (lay.cache + cl - 1) / cl;
    a.o_acc = oacc;
    CK_CUDA(launch_attention(a, s, cl));
    // phases 10-11: output rows, residual (and its squares for the feed-forward norm)
    int64_t* next = cur == x ? xb : x;
    MatrowParams po = {};
    po.W = W.wo;
    po.scale = W.so;
    po.grouped = 1;
    po.pitch = m->pitch_d;
    po.rows = c.dim;
    po.cols = c.dim;
    po.pro = kProPlain;
    po.in = o;
    po.in_acc = oacc;  // when set: o is written from the sums by block 0
    po.in_out = o;
    po.epi = kEpiStore;
    po.out = y;
    po.resid_in = cur;
    po.resid_out = next;
    po.ss_out = ss + 2 * l + 1;
    po.state = st;
    CK_CUDA(launch_matrow(po, s, m->num_sms));
    cur = next;
    // phases 12-14: feed-forward norm, gate and up, SiLU gating
    MatrowParams pg = {};
    pg.W = W.w13;
    pg.scale = W.s13;
    pg.grouped = 1;
    pg.pitch = m->pitch_d;
    pg.rows = 2 * c.hidden;
    pg.cols = c.dim;
    pg.pro = kProNorm;
    pg.in = cur;
    pg.ss_in = ss + 2 * l + 1;
    pg.norm_w = W.ffn_norm;
    pg.epi = kEpiSiLU;
    pg.out = hbuf;
    pg.silu_tab = m->silu_tab;
    pg.acc_clear = oacc;
    pg.acc_words = c.dim;
    pg.planes_out = hplanes;
    pg.planes_pitch = m->pitch_h;
    pg.parts_out = hparts;
    pg.state = st;
    CK_CUDA(launch_matrow(pg, s, m->num_sms));
    // phases 15-16: down rows, residual (and its squares for the next norm)
    next = cur == x ? xb : x;
    MatrowParams pd = {};
    pd.W = W.w2;
    pd.scale = W.s2;
    pd.grouped = 1;
    pd.pitch = m->pitch_h;
    pd.rows = c.dim;
    pd.cols = c.hidden;
    pd.pro = kProPlain;
    pd.in = hbuf;
    pd.in_planes = hplanes;  // when set: the planes and partials replace reading hbuf
    pd.parts_in = hparts;
    pd.nparts = gu_grid;
    pd.epi = kEpiStore;
    pd.out = y;
    pd.resid_in = cur;
    pd.resid_out = next;
    pd.ss_out = ss + 2 * (l + 1);
    pd.state = st;
    CK_CUDA(launch_matrow(pd, s, m->num_sms));
    cur = next;
  }
  if (cur != x) return CK_INVALID_STATE;  // an even number of residual flips, by construction
  if (generating) {
    // phases 17-18: final norm, classifier
    MatrowParams pc = {};
    pc.W = m->cls;
    pc.scale = m->cls_scale;
    pc.grouped = 1;
    pc.pitch = m->pitch_d;
    pc.rows = c.vocab;
    pc.cols = c.dim;
    pc.pro = kProNorm;
    pc.in = x;
    pc.ss_in = ss + 2 * c.layers;
    pc.norm_w = m->final_norm;
    pc.epi = kEpiStore;
    pc.out = logits;
    pc.state = st;
    CK_CUDA(launch_matrow(pc, s, m->num_sms));
    k_sample_finish<<<1, kArgThreads, 0, s>>>(st, lay.out, logits, c.vocab, m->exp_tab);  // phase 19
  } else {
    k_finish_prompt<<<1, 32, 0, s>>>(st);
  }
  CK_CUDA(cudaGetLastError());
  return CK_OK;
}

// Launch plan of the one-position kernel for a state, or false when the model or state is
// outside what it supports (then the phase-by-phase kernels run instead).  state_work: the
// kernel's scratch is the state's work region, which must then hold it (the allocation-free
// entry keeps its scratch elsewhere and checks its own limit).
bool plan_step(const ck_model* m, const StateLayout& lay, StepParams* sp, int* grid, size_t* smem,
               bool state_work = true) {
  const ck_config& c = m->cfg;
  if (c.heads > 1000) return false;
  const int G = m->num_sms < 768 ? m->num_sms : 768;
  const uint32_t gh = c.heads >= (uint32_t)G ? 1u : (uint32_t)G / c.heads;
  if (c.heads * gh > (uint32_t)G) return false;
  const uint64_t hd = m->head_dim;
  // attention: every CTA of a head scores all positions up to att_full (the head's keys are
  // then read by each of its CTAs, from L2 after the first); beyond, the scoring is split
  const uint32_t att_def = m->att_full ? m->att_full : (uint32_t)(16384 / hd);
  const uint32_t att_full = gh == 1 ? lay.cache : std::min<uint32_t>(lay.cache, att_def);
  const uint64_t chunk = (lay.cache + gh - 1) / gh;
  const uint64_t nscore = std::max<uint64_t>(chunk, att_full);
  const uint64_t attn = 8ull * (hd * (1 + kStepWarps) + kStepWarps + nscore);
  const uint64_t max_pitch = std::max(m->pitch_d, m->pitch_h);
  // byte planes in shared memory: at least four limbs of the widest input, eight of a
  // dim-wide one when they fit in 48 KB; planes beyond go to a global copy (rare)
  const uint64_t planes = std::max<uint64_t>(4 * max_pitch, std::min<uint64_t>(8ull * m->pitch_d, 48 * 1024));
  // most rows a block takes in one matrix (whole pairs split over the grid), plus slack
  const uint64_t max_rows = std::max<uint64_t>(
      std::max<uint64_t>((uint64_t)c.dim + 2 * (uint64_t)m->kv_dim, 2 * (uint64_t)c.hidden),
      std::max<uint64_t>((uint64_t)c.dim, (uint64_t)c.vocab));
  const uint64_t scale_cap = 2 * (((max_rows + 1) / 2 + G - 1) / G) + 2;
  // X region: planes, row scales, rotary row, residual slice, next norm's weights slice
  const uint64_t x_vslice = (planes + 4 * scale_cap + 4 * hd + 15) & ~15ull;
  const uint64_t x_wslice = x_vslice + 8 * scale_cap;
  const uint64_t xb = (std::max<uint64_t>(attn, x_wslice + 4 * scale_cap) + 15) & ~15ull;
  const uint64_t red = (uint64_t)step_red_bytes();
  const uint64_t avail = (uint64_t)m->step_smem;
  if (avail < xb + red + 2 * (kStageBytes + 16) + 16) return false;
  uint64_t ns = (avail - xb - red - 16) / (kStageBytes + 16);
  if (ns > kMaxSlots) ns = kMaxSlots;
  if (m->max_slots && ns > m->max_slots) ns = m->max_slots;
  if (ns < 2) return false;
  // work region: cleared counters and sums, attention partials, classifier candidates,
  // attention accumulators, the three plane buffers of the phase inputs
  const uint64_t off_hsync = 256, off_hfin = off_hsync + 4ull * c.heads;
  const uint64_t zero_bytes = (off_hfin + 4ull * c.heads + 255) & ~255ull;
  const uint64_t off_part = zero_bytes;
  const uint64_t off_cand = off_part + 16ull * c.heads * gh;
  const uint64_t off_oacc = (off_cand + 16ull * G + 255) & ~255ull;
  const uint64_t off_vbuf = (off_oacc + 8ull * c.dim + 255) & ~255ull;
  const uint64_t work_need = off_vbuf + 3 * 8 * max_pitch;
  const uint64_t work_bytes = lay.k - lay.scores;
  if (state_work && work_need > work_bytes) return false;
  StepParams& p = *sp;
  p = StepParams{};
  p.off_prompt = lay.prompt; p.off_out = lay.out; p.off_x = lay.x; p.off_xb = lay.xb; p.off_q = lay.q;
  p.off_o = lay.o; p.off_y = lay.y; p.off_h = lay.h; p.off_logits = lay.logits;
  p.off_work = lay.scores; p.off_k = lay.k; p.off_v = lay.v;
  p.cache = lay.cache;
  p.dim = c.dim; p.hidden = c.hidden; p.layers = c.layers; p.heads = c.heads; p.kv_heads = c.kv_heads;
  p.vocab = c.vocab; p.hd = m->head_dim; p.kv_dim = m->kv_dim; p.pitch_d = m->pitch_d;
  p.pitch_h = m->pitch_h; p.inv_sqrt = m->inv_sqrt;
  p.gh = gh; p.att_full = att_full; p.ns = (uint32_t)ns; p.x_bytes = (uint32_t)xb;
  p.pf_bytes = m->pf_kb * 1024u;  // 0 (the default): none
  p.sync_polls = m->sync_polls;   // 0 (the default): the kernel's own limit
  p.planes_bytes = (uint32_t)planes;
  p.zero_bytes = (uint32_t)zero_bytes; p.off_hsync = (uint32_t)off_hsync; p.off_hfin = (uint32_t)off_hfin;
  p.off_part = off_part; p.off_cand = off_cand; p.off_oacc = off_oacc; p.off_vbuf = off_vbuf;
  p.vbuf_pitch = (uint32_t)max_pitch;
  p.x_vslice = (uint32_t)x_vslice; p.x_wslice = (uint32_t)x_wslice;
  p.scale_cap = (uint32_t)scale_cap;
  p.div_dim = make_invdiv(c.dim);
  p.div_hidden = make_invdiv(c.hidden);
  p.layers_tab = m->dev_layers;
  p.embed = m->embed; p.embed_scale = m->embed_scale; p.cls = m->cls; p.cls_scale = m->cls_scale;
  p.final_norm = m->final_norm; p.rope = m->rope; p.exp_tab = m->exp_tab; p.silu_tab = m->silu_tab;
  *grid = G;
  *smem = xb + red + ns * kStageBytes + 16 * ns + 16;  // + the plane-copy barrier
  return step_blocks_per_sm(*smem) >= 1;  // every block must be resident for the grid barriers
}

// Bytes of the work region the one-position kernel uses for a plan.
size_t step_work_bytes(const StepParams& p) { return p.off_vbuf + 3ull * 8 * p.vbuf_pitch; }

int enqueue_step(const ck_model* m, uint8_t* st, const StateLayout& lay, bool generating,
                 cudaStream_t s) {
  StepParams p;
  int grid;
  size_t smem;
  if (!plan_step(m, lay, &p, &grid, &smem)) return CK_INVALID_ARGUMENT;
  p.st = st;
  p.generating = generating ? 1u : 0u;
  CK_CUDA(cudaMemsetAsync(st + lay.scores, 0, p.zero_bytes, s));  // counters and per-vector sums
  CK_CUDA(launch_step(p, s, grid, smem));
  return CK_OK;
}

// CK_PATH_AUTO takes the phase kernels: with programmatic dependent launch they are faster
// than the persistent kernel on every model measured (7B and 1B shapes from 64 to 8K cached
// positions, and the small test models).
int resolve_path(const ck_model* m, const StateLayout& lay) {
  if (m->path != CK_PATH_STEP) return CK_PATH_KERNELS;
  StepParams p;
  int grid;
  size_t smem;
  return plan_step(m, lay, &p, &grid, &smem) ? CK_PATH_STEP : -1;
}

int get_graph(ck_model* m, void* dev_state, size_t len, const StateLayout& lay, bool generating,
              cudaGraphExec_t* out) {
  const int path = resolve_path(m, lay);
  if (path < 0) return CK_INVALID_ARGUMENT;
  for (auto& g : m->graphs)
    if (g.state == dev_state && g.len == len && g.generating == generating && g.path == path) {
      *out = g.exec;
      return CK_OK;
    }
  if (m->graphs.size() >= 16) {  // bounded cache: drop the oldest pair
    cudaGraphExecDestroy(m->graphs.front().exec);
    m->graphs.erase(m->graphs.begin());
  }
  CK_CUDA(cudaStreamBeginCapture(m->capture, cudaStreamCaptureModeThreadLocal));
  int rc = path == CK_PATH_STEP
               ? enqueue_step(m, static_cast<uint8_t*>(dev_state), lay, generating, m->capture)
               : enqueue_position(m, static_cast<uint8_t*>(dev_state), lay, generating, m->capture);
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(m->capture, &graph);
  if (rc) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (e != cudaSuccess) return CK_CUDA_ERROR;
  cudaGraphExec_t exec;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return CK_CUDA_ERROR;
  m->graphs.push_back({dev_state, len, generating, path, exec});
  *out = exec;
  return CK_OK;
}

PrefillModel prefill_model(const ck_model* m) {
  PrefillModel pm;
  pm.cfg = m->cfg;
  pm.head_dim = m->head_dim;
  pm.kv_dim = m->kv_dim;
  pm.inv_sqrt = m->inv_sqrt;
  pm.pitch_d = m->pitch_d;
  pm.pitch_h = m->pitch_h;
  pm.embed = m->embed;
  pm.embed_scale = m->embed_scale;
  pm.layers = m->layers.data();
  pm.rope = m->rope;
  pm.exp_tab = m->exp_tab;
  pm.silu_tab = m->silu_tab;
  pm.cls = m->cls;
  pm.cls_scale = m->cls_scale;
  pm.final_norm = m->final_norm;
  pm.num_sms = m->num_sms;
  return pm;
}

void drop_batch_graphs(ck_model* m) {
  for (auto& g : m->bgraphs) cudaGraphExecDestroy(g.exec);
  m->bgraphs.clear();
}

// The batched kernels' scratch, laid out for at least `rows` rows.
int ensure_batch_work(ck_model* m, uint32_t rows) {
  if (!m->pf_configured) {
    CK_CUDA(configure_prefill((size_t)m->smem_optin));
    m->pf_configured = true;
  }
  if (m->pf_work && m->pf_wcap >= rows) return CK_OK;
  const uint32_t cap = std::max(rows, m->pf_wcap);
  const size_t need = prefill_work_bytes(prefill_model(m), cap);
  drop_batch_graphs(m);  // they point into the scratch
  if (m->pf_work) CK_CUDA(cudaFree(m->pf_work));
  m->pf_work = nullptr;
  m->pf_bytes = 0;
  m->pf_wcap = 0;
  CK_CUDA(cudaMalloc(&m->pf_work, need));
  m->pf_bytes = need;
  m->pf_wcap = cap;
  return CK_OK;
}

// The batched pass's kernels for n rows and a position bound, as a CUDA graph (captured at
// first use, kept in a small cache): one launch per pass instead of one per kernel.
int get_batch_graph(ck_model* m, uint32_t n, uint32_t max_positions, cudaGraphExec_t* out) {
  for (auto& g : m->bgraphs)
    if (g.n == n && g.max_positions == max_positions && g.work == m->pf_work && g.cap == m->pf_wcap) {
      *out = g.exec;
      return CK_OK;
    }
  if (m->bgraphs.size() >= 8) {
    cudaGraphExecDestroy(m->bgraphs.front().exec);
    m->bgraphs.erase(m->bgraphs.begin());
  }
  CK_CUDA(cudaStreamBeginCapture(m->capture, cudaStreamCaptureModeThreadLocal));
  const cudaError_t ek = enqueue_batch_kernels(prefill_model(m), n, max_positions, m->pf_work, m->pf_wcap,
                                               m->capture);
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(m->capture, &graph);
  if (ek != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    return CK_CUDA_ERROR;
  }
  if (e != cudaSuccess) return CK_CUDA_ERROR;
  cudaGraphExec_t exec;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return CK_CUDA_ERROR;
  m->bgraphs.push_back({n, max_positions, m->pf_work, m->pf_wcap, exec});
  *out = exec;
  return CK_OK;
}

// Positions pos .. pos+P-1 layer by layer.  CK_INVALID_ARGUMENT: the batched kernels do not
// handle this model or cache (the caller runs the positions one by one instead).
int prefill_chunk(ck_model* m, uint8_t* st, const StateLayout& lay, uint32_t pos, uint32_t P,
                  cudaStream_t s) {
  const PrefillModel pm = prefill_model(m);
  if (!prefill_supported(pm, lay.cache, (size_t)m->smem_optin)) return CK_INVALID_ARGUMENT;
  const int rc = ensure_batch_work(m, m->pf_cap);
  if (rc) return rc;
  CK_CUDA(enqueue_prefill(pm, st, lay, pos, P, m->pf_work, m->pf_wcap, s));
  return CK_OK;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

const char* ck_version(void) { return "libck 0.1 (sm_103a)"; }

uint64_t ck_host_isqrt(uint64_t v) { return isqrt_u64(v); }

uint64_t ck_host_probability(uint64_t e, uint64_t z) {
  if (z == 0) return 0;
  return div_by_estimate(e << 24, z, rcp_estimate((float)z));
}

int64_t ck_host_div_trunc(int64_t n, uint32_t d) {
  if (d == 0) return 0;
  return sdiv_trunc(n, make_invdiv_fast(d));
}

int ck_model_size(const void* artifact, size_t len, size_t* dev_bytes) {
  if (!dev_bytes) return CK_INVALID_ARGUMENT;
  Parsed P;
  int rc = parse_artifact(artifact, len, &P);
  if (rc) return rc;
  *dev_bytes = plan_device(P.cfg, P.flags & 1u).total;
  return CK_OK;
}

int ck_load_model(const void* artifact, size_t len, void* dev_mem, size_t dev_len, void* stream,
                  ck_model** out) {
  if (!out || !dev_mem) return CK_INVALID_ARGUMENT;
  *out = nullptr;
  if (reinterpret_cast<uintptr_t>(dev_mem) % 256) return CK_INVALID_ARGUMENT;
  Parsed P;
  int rc = parse_artifact(artifact, len, &P);
  if (rc) return rc;
  const ck_config& c = P.cfg;
  const bool tied = P.flags & 1u;
  DevPlan D = plan_device(c, tied);
  if (dev_len < D.total) return CK_BUFFER_TOO_SMALL;
  cudaStream_t s = S(stream);
  uint8_t* dv = static_cast<uint8_t*>(dev_mem);
  const uint32_t pd = pad128(c.dim), ph = pad128(c.hidden), hd = c.dim / c.heads;
  const uint32_t kv = hd * c.kv_heads;
  CK_CUDA(cudaMemsetAsync(dv, 0, D.total, s));
  auto T = [&](uint32_t i) { return P.t[i]; };
  std::vector<uint8_t> stage;
  // a row-major source matrix of `cols`-byte rows
  auto plain = [](const uint8_t* base, uint32_t cols) {
    return [base, cols](uint32_t r) { return base + (size_t)r * cols; };
  };
  CK_CUDA(upload_grouped(dv + D.embed, c.vocab, c.dim, pd, plain(T(0), c.dim), stage, s));
  CK_CUDA(cudaMemcpyAsync(dv + D.embed_scale, T(1), 4ull * c.vocab, cudaMemcpyHostToDevice, s));
  if (!tied) {
    CK_CUDA(upload_grouped(dv + D.cls, c.vocab, c.dim, pd, plain(T(3), c.dim), stage, s));
    CK_CUDA(cudaMemcpyAsync(dv + D.cls_scale, T(4), 4ull * c.vocab, cudaMemcpyHostToDevice, s));
  }
  CK_CUDA(cudaMemcpyAsync(dv + D.final_norm, T(2), 4ull * c.dim, cudaMemcpyHostToDevice, s));
  CK_CUDA(cudaMemcpyAsync(dv + D.rope, T(5), 4ull * c.context * hd, cudaMemcpyHostToDevice, s));
  CK_CUDA(cudaMemcpyAsync(dv + D.exp_tab, T(6), 4ull * kTable, cudaMemcpyHostToDevice, s));
  CK_CUDA(cudaMemcpyAsync(dv + D.silu_tab, T(7), 4ull * kTable, cudaMemcpyHostToDevice, s));
  for (uint32_t l = 0; l < c.layers; ++l) {
    const DevPlan::L& L = D.layers[l];
    const uint32_t b = 8 + 16 * l;
    CK_CUDA(cudaMemcpyAsync(dv + L.an, T(b + 0), 4ull * c.dim, cudaMemcpyHostToDevice, s));
    // Q rows, then K rows, then V rows as one matrix
    const uint8_t *wq = T(b + 1), *wk = T(b + 3), *wv = T(b + 5);
    const uint32_t dim = c.dim;
    CK_CUDA(upload_grouped(dv + L.wqkv, c.dim + 2 * kv, c.dim, pd,
                           [=](uint32_t r) {
                             return r < dim ? wq + (size_t)r * dim
                                            : r < dim + kv ? wk + (size_t)(r - dim) * dim
                                                           : wv + (size_t)(r - dim - kv) * dim;
                           },
                           stage, s));
    CK_CUDA(cudaMemcpyAsync(dv + L.sqkv, T(b + 2), 4ull * c.dim, cudaMemcpyHostToDevice, s));
    CK_CUDA(cudaMemcpyAsync(dv + L.sqkv + 4ull * c.dim, T(b + 4), 4ull * kv, cudaMemcpyHostToDevice, s));
    CK_CUDA(cudaMemcpyAsync(dv + L.sqkv + 4ull * (c.dim + kv), T(b + 6), 4ull * kv,
                            cudaMemcpyHostToDevice, s));
    CK_CUDA(upload_grouped(dv + L.wo, c.dim, c.dim, pd, plain(T(b + 7), c.dim), stage, s));
    CK_CUDA(cudaMemcpyAsync(dv + L.so, T(b + 8), 4ull * c.dim, cudaMemcpyHostToDevice, s));
    CK_CUDA(cudaMemcpyAsync(dv + L.fn, T(b + 9), 4ull * c.dim, cudaMemcpyHostToDevice, s));
    // gate rows to even rows, up rows to odd rows (and their scales likewise)
    const uint8_t *wg = T(b + 10), *wu = T(b + 12);
    CK_CUDA(upload_grouped(dv + L.w13, 2 * c.hidden, c.dim, pd,
                           [=](uint32_t r) { return ((r & 1) ? wu : wg) + (size_t)(r >> 1) * dim; },
                           stage, s));
    CK_CUDA(cudaMemcpy2DAsync(dv + L.s13, 8, T(b + 11), 4, 4, c.hidden, cudaMemcpyHostToDevice, s));
    CK_CUDA(cudaMemcpy2DAsync(dv + L.s13 + 4, 8, T(b + 13), 4, 4, c.hidden, cudaMemcpyHostToDevice, s));
    CK_CUDA(upload_grouped(dv + L.w2, c.dim, c.hidden, ph, plain(T(b + 14), c.hidden), stage, s));
    CK_CUDA(cudaMemcpyAsync(dv + L.s2, T(b + 15), 4ull * c.dim, cudaMemcpyHostToDevice, s));
  }
  CK_CUDA(cudaStreamSynchronize(s));

  ck_model* m = new (std::nothrow) ck_model();
  if (!m) return CK_CUDA_ERROR;
  m->cfg = c;
  m->head_dim = hd;
  m->kv_dim = kv;
  m->inv_sqrt = P.inv_sqrt;
  m->flags = P.flags;
  m->pitch_d = pd;
  m->pitch_h = ph;
  m->dev = dv;
  m->dev_len = dev_len;
  m->embed = dv + D.embed;
  m->embed_scale = reinterpret_cast<const uint32_t*>(dv + D.embed_scale);
  m->cls = dv + D.cls;
  m->cls_scale = reinterpret_cast<const uint32_t*>(dv + D.cls_scale);
  m->final_norm = reinterpret_cast<const int32_t*>(dv + D.final_norm);
  m->rope = reinterpret_cast<const int32_t*>(dv + D.rope);
  m->exp_tab = reinterpret_cast<const uint32_t*>(dv + D.exp_tab);
  m->silu_tab = reinterpret_cast<const int32_t*>(dv + D.silu_tab);
  m->scratch = reinterpret_cast<uint32_t*>(dv + D.scratch);
  m->layers.resize(c.layers);
  for (uint32_t l = 0; l < c.layers; ++l) {
    const DevPlan::L& L = D.layers[l];
    DevLayer& W = m->layers[l];
    W.wqkv = dv + L.wqkv;
    W.sqkv = reinterpret_cast<const uint32_t*>(dv + L.sqkv);
    W.wo = dv + L.wo;
    W.so = reinterpret_cast<const uint32_t*>(dv + L.so);
    W.w13 = dv + L.w13;
    W.s13 = reinterpret_cast<const uint32_t*>(dv + L.s13);
    W.w2 = dv + L.w2;
    W.s2 = reinterpret_cast<const uint32_t*>(dv + L.s2);
    W.attn_norm = reinterpret_cast<const int32_t*>(dv + L.an);
    W.ffn_norm = reinterpret_cast<const int32_t*>(dv + L.fn);
  }
  m->dev_layers = reinterpret_cast<DevLayer*>(dv + D.table);
  m->path = CK_PATH_AUTO;
  m->max_slots = 0;
  m->att_full = 0;
  m->pf_kb = 0;
  m->pf_cap = kDefaultPrefillChunk;
  m->pf_work = nullptr;
  m->pf_bytes = 0;
  m->pf_wcap = 0;
  m->pf_configured = false;
  if (cudaMemcpyAsync(m->dev_layers, m->layers.data(), sizeof(DevLayer) * c.layers,
                      cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    delete m;
    return CK_CUDA_ERROR;
  }
  if (configure_matrow() != cudaSuccess || configure_attention() != cudaSuccess) {
    delete m;
    return CK_CUDA_ERROR;
  }
  if (cudaGetDevice(&m->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&m->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, m->device) !=
          cudaSuccess ||
      configure_step((size_t)m->smem_optin, &m->step_smem) != cudaSuccess ||
      cudaStreamCreateWithFlags(&m->capture, cudaStreamNonBlocking) != cudaSuccess) {
    delete m;
    return CK_CUDA_ERROR;
  }
  *out = m;
  return CK_OK;
}

int ck_set_path(ck_model* m, int path) {
  if (!m || path < CK_PATH_AUTO || path > CK_PATH_KERNELS) return CK_INVALID_ARGUMENT;
  m->path = path;
  return CK_OK;
}

int ck_set_step_slots(ck_model* m, uint32_t max_slots) {
  if (!m || max_slots == 1 || max_slots > kMaxSlots) return CK_INVALID_ARGUMENT;
  m->max_slots = max_slots;
  for (auto& g : m->graphs) cudaGraphExecDestroy(g.exec);  // plans change: rebuild graphs
  m->graphs.clear();
  return CK_OK;
}

int ck_set_step_wait_limit(ck_model* m, uint32_t polls) {
  if (!m) return CK_INVALID_ARGUMENT;
  m->sync_polls = polls;
  for (auto& g : m->graphs) cudaGraphExecDestroy(g.exec);  // plans change: rebuild graphs
  m->graphs.clear();
  return CK_OK;
}

int ck_set_step_prefetch(ck_model* m, uint32_t kb_per_block) {
  if (!m || kb_per_block > 4096) return CK_INVALID_ARGUMENT;
  m->pf_kb = kb_per_block;
  for (auto& g : m->graphs) cudaGraphExecDestroy(g.exec);
  m->graphs.clear();
  return CK_OK;
}

int ck_set_attention_split(ck_model* m, uint32_t positions) {
  if (!m) return CK_INVALID_ARGUMENT;
  m->att_full = positions;
  for (auto& g : m->graphs) cudaGraphExecDestroy(g.exec);
  m->graphs.clear();
  return CK_OK;
}

int ck_model_config(const ck_model* m, ck_config* out) {
  if (!m || !out) return CK_INVALID_ARGUMENT;
  *out = m->cfg;
  return CK_OK;
}

int ck_set_prefill(ck_model* m, uint32_t positions) {
  if (!m || positions > kMaxPrefillChunk) return CK_INVALID_ARGUMENT;
  m->pf_cap = positions;
  drop_batch_graphs(m);
  if (m->pf_work) cudaFree(m->pf_work);  // resized at next use
  m->pf_work = nullptr;
  m->pf_bytes = 0;
  m->pf_wcap = 0;
  return CK_OK;
}

void ck_free_model(ck_model* m) {
  if (!m) return;
  drop_batch_graphs(m);
  if (m->pf_work) cudaFree(m->pf_work);
  for (auto& g : m->graphs) cudaGraphExecDestroy(g.exec);
  if (m->capture) cudaStreamDestroy(m->capture);
  delete m;
}

int ck_state_size(const ck_model* m, uint32_t n_prompt, uint32_t max_tokens, size_t* out) {
  if (!m || !out) return CK_INVALID_ARGUMENT;
  if (!n_prompt || !max_tokens || max_tokens > m->cfg.context) return CK_INVALID_PROMPT;
  if ((uint64_t)n_prompt + max_tokens - 1 > m->cfg.context) return CK_CONTEXT_EXCEEDED;
  *out = state_layout(m->cfg, n_prompt, max_tokens).size;
  return CK_OK;
}

int ck_init_state(const ck_model* m, void* dev_state, size_t len, const uint32_t* host_ids,
                  uint32_t n_ids, uint32_t max_tokens, uint32_t temperature_q16, uint64_t seed,
                  uint32_t flags, void* stream) {
  if (!m || !dev_state || (n_ids && !host_ids)) return CK_INVALID_ARGUMENT;
  if (reinterpret_cast<uintptr_t>(dev_state) % 256) return CK_INVALID_STATE;
  if (!n_ids || !max_tokens || max_tokens > m->cfg.context) return CK_INVALID_PROMPT;
  if (temperature_q16 > kMaxTemperature) return CK_INVALID_PROMPT;
  for (uint32_t i = 0; i < n_ids; ++i)
    if (host_ids[i] >= m->cfg.vocab) return CK_INVALID_PROMPT;
  if ((uint64_t)n_ids + max_tokens - 1 > m->cfg.context) return CK_CONTEXT_EXCEEDED;
  const StateLayout lay = state_layout(m->cfg, n_ids, max_tokens);
  if (len != lay.size) return CK_BUFFER_TOO_SMALL;
  std::vector<uint8_t> h(lay.x, 0);  // header, prompt ids and output tokens
  memcpy(h.data(), "CKSTATE1", 8);
  auto w32 = [&](uint32_t off, uint32_t v) { memcpy(h.data() + off, &v, 4); };
  auto w64 = [&](uint32_t off, uint64_t v) { memcpy(h.data() + off, &v, 8); };
  w32(kHPhase, CK_PHASE_RUNNING);
  w32(kHNPrompt, n_ids);
  w32(kHMaxTok, max_tokens);
  w32(kHCache, lay.cache);
  w32(kHFlags, flags);
  w32(kHTemp, temperature_q16);
  w32(kHLastTok, 0xFFFFFFFFu);
  w64(kHSeed, seed ? seed : kZeroSeedState);  // the generator's first state
  w64(kHErrKey, kNoError);
  for (int i = 0; i < 7; ++i) w32(kHConfig + 4 * i, (&m->cfg.dim)[i]);
  memcpy(h.data() + lay.prompt, host_ids, 4ull * n_ids);
  cudaStream_t s = S(stream);
  CK_CUDA(cudaMemsetAsync(dev_state, 0, len, s));
  CK_CUDA(cudaMemcpyAsync(dev_state, h.data(), h.size(), cudaMemcpyHostToDevice, s));
  CK_CUDA(cudaStreamSynchronize(s));
  return CK_OK;
}

int ck_turn(ck_model* m, void* dev_state, size_t len, uint32_t n_positions, void* stream,
            ck_turn_result* out) {
  if (!m || !dev_state || !out) return CK_INVALID_ARGUMENT;
  memset(out, 0, sizeof(*out));
  out->token = 0xFFFFFFFFu;
  if (reinterpret_cast<uintptr_t>(dev_state) % 256) return CK_INVALID_STATE;
  cudaStream_t s = S(stream);
  HostHeader h0;
  int rc = read_header(dev_state, &h0, s);
  if (rc) return rc;
  StateLayout lay;
  rc = check_state(m, dev_state, len, h0, &lay);
  if (rc) return rc;
  if (h0.u32(kHPhase) != CK_PHASE_RUNNING) return CK_INVALID_STATE;
  const uint32_t pos0 = h0.u32(kHPosition), np = h0.u32(kHNPrompt);
  if (pos0 >= lay.cache) return CK_INVALID_STATE;
  uint32_t n = n_positions;
  if (n > lay.cache - pos0) n = lay.cache - pos0;
  for (uint32_t i = 0; i < n;) {
    const uint32_t pos = pos0 + i;
    // two or more prompt positions that generate no token: layer-major, in chunks
    const uint32_t run = pos + 1 < np ? std::min(np - 1 - pos, n - i) : 0u;
    if (run >= 2 && m->pf_cap >= 2) {
      const uint32_t P = std::min(run, m->pf_cap);
      rc = prefill_chunk(m, static_cast<uint8_t*>(dev_state), lay, pos, P, s);
      if (rc != CK_OK && rc != CK_INVALID_ARGUMENT) return rc;
      if (rc == CK_OK) {
        i += P;
        continue;
      }
    }
    const bool generating = pos + 1 >= np;
    cudaGraphExec_t exec;
    rc = get_graph(m, dev_state, len, lay, generating, &exec);
    if (rc) return rc;
    CK_CUDA(cudaGraphLaunch(exec, s));
    ++i;
  }
  HostHeader h1;
  rc = read_header(dev_state, &h1, s);
  if (rc) return rc;
  const bool failed = h1.u32(kHPhase) == CK_PHASE_FAILED;
  uint64_t turns = h1.u64(kHTurns) + 1;
  CK_CUDA(cudaMemcpyAsync(static_cast<uint8_t*>(dev_state) + kHTurns, &turns, 8,
                          cudaMemcpyHostToDevice, s));
  CK_CUDA(cudaStreamSynchronize(s));
  out->generated = h1.u32(kHGenerated);
  out->generated_this_turn = out->generated - h0.u32(kHGenerated);
  if (out->generated_this_turn) out->token = h1.u32(kHLastTok);
  out->work = h1.u32(kHPosition) - pos0 + (failed ? 1u : 0u);
  out->complete = h1.u32(kHPhase) != CK_PHASE_RUNNING;
  const uint64_t key = h1.u64(kHErrKey);
  if (key != kNoError) {
    out->err_position = (uint32_t)(key >> 44);
    out->err_layer = (uint32_t)(key >> 32) & 0xFFFu;
    out->err_phase = (uint32_t)(key >> 24) & 0xFFu;
    out->err_element = (uint32_t)key & 0xFFFFFFu;
  }
  return failed ? (int)h1.u32(kHError) : CK_OK;
}

int ck_turn_batch(ck_model* m, void* const* dev_states, const size_t* lens, uint32_t n_states,
                  void* stream, ck_turn_result* out, int* rcs) {
  if (!m || !dev_states || !lens || !out || !rcs || n_states == 0 || n_states > kMaxPrefillChunk)
    return CK_INVALID_ARGUMENT;
  for (uint32_t i = 0; i < n_states; ++i)
    if (!dev_states[i]) return CK_INVALID_ARGUMENT;
  {
    std::vector<void*> sorted(dev_states, dev_states + n_states);
    std::sort(sorted.begin(), sorted.end());
    if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end()) return CK_INVALID_ARGUMENT;
  }
  for (uint32_t i = 0; i < n_states; ++i) {
    memset(&out[i], 0, sizeof(out[i]));
    out[i].token = 0xFFFFFFFFu;
    rcs[i] = CK_OK;
  }
  cudaStream_t s = S(stream);
  const PrefillModel pm = prefill_model(m);
  int rc = ensure_batch_work(m, n_states);
  if (rc) return rc;
  // the states that can take a position: aligned, this model's, running, with a position left
  std::vector<uint32_t> idx;
  std::vector<uint8_t*> ptrs;
  for (uint32_t i = 0; i < n_states; ++i) {
    if (reinterpret_cast<uintptr_t>(dev_states[i]) % 256) {
      rcs[i] = CK_INVALID_STATE;
      continue;
    }
    idx.push_back(i);
    ptrs.push_back(static_cast<uint8_t*>(dev_states[i]));
  }
  std::vector<uint8_t> h0(kHeaderBytes * idx.size() + 1), h1(h0.size());
  if (!idx.empty())
    CK_CUDA(batch_gather_headers(pm, ptrs.data(), (uint32_t)idx.size(), m->pf_work, m->pf_wcap, h0.data(), s));
  std::vector<RowDesc> rows;
  std::vector<uint32_t> row_of;  // index into dev_states of each row
  uint32_t max_positions = 1, max_cache = 1;
  for (size_t j = 0; j < idx.size(); ++j) {
    const uint32_t i = idx[j];
    HostHeader h;
    memcpy(h.b, h0.data() + kHeaderBytes * j, kHeaderBytes);
    StateLayout lay;
    if (check_state(m, dev_states[i], lens[i], h, &lay) != CK_OK || h.u32(kHPhase) != CK_PHASE_RUNNING ||
        h.u32(kHPosition) >= lay.cache) {
      rcs[i] = CK_INVALID_STATE;
      continue;
    }
    if (!prefill_supported(pm, lay.cache, (size_t)m->smem_optin)) return CK_INVALID_ARGUMENT;
    RowDesc r = {};
    r.st = static_cast<uint8_t*>(dev_states[i]);
    r.pos = h.u32(kHPosition);
    r.cache = lay.cache;
    r.np = h.u32(kHNPrompt);
    r.generating = r.pos + 1 >= r.np ? 1u : 0u;
    r.off_prompt = lay.prompt;
    r.off_out = lay.out;
    r.off_x = lay.x;
    r.off_logits = lay.logits;
    r.off_k = lay.k;
    r.off_v = lay.v;
    rows.push_back(r);
    row_of.push_back(i);
    max_positions = std::max(max_positions, r.pos + 1);
    max_cache = std::max(max_cache, r.cache);
    out[i].generated = h.u32(kHGenerated);  // before; replaced below
  }
  if (!rows.empty()) {
    // the position bound rounded up to a multiple of 128 (within the largest cache: the
    // attention's shared memory is checked for every row's cache), so that one graph serves
    // many passes
    const uint32_t bound = std::min(max_cache, (max_positions + 127) / 128 * 128);
    CK_CUDA(upload_batch_rows(pm, rows.data(), (uint32_t)rows.size(), m->pf_work, m->pf_wcap, s));
    cudaGraphExec_t exec;
    rc = get_batch_graph(m, (uint32_t)rows.size(), bound, &exec);
    if (rc) return rc;
    CK_CUDA(cudaGraphLaunch(exec, s));
    std::vector<uint8_t*> rptrs;
    for (const RowDesc& r : rows) rptrs.push_back(r.st);
    CK_CUDA(batch_gather_headers(pm, rptrs.data(), (uint32_t)rows.size(), m->pf_work, m->pf_wcap, h1.data(), s));
  }
  int first = CK_OK;
  for (size_t j = 0; j < rows.size(); ++j) {
    const uint32_t i = row_of[j];
    HostHeader h;
    memcpy(h.b, h1.data() + kHeaderBytes * j, kHeaderBytes);
    const bool failed = h.u32(kHPhase) == CK_PHASE_FAILED;
    ck_turn_result& o = out[i];
    const uint32_t gen0 = o.generated;
    o.generated = h.u32(kHGenerated);
    o.generated_this_turn = o.generated - gen0;
    if (o.generated_this_turn) o.token = h.u32(kHLastTok);
    o.work = h.u32(kHPosition) - rows[j].pos + (failed ? 1u : 0u);
    o.complete = h.u32(kHPhase) != CK_PHASE_RUNNING;
    const uint64_t key = h.u64(kHErrKey);
    if (key != kNoError) {
      o.err_position = (uint32_t)(key >> 44);
      o.err_layer = (uint32_t)(key >> 32) & 0xFFFu;
      o.err_phase = (uint32_t)(key >> 24) & 0xFFu;
      o.err_element = (uint32_t)key & 0xFFFFFFu;
    }
    rcs[i] = failed ? (int)h.u32(kHError) : CK_OK;
  }
  for (uint32_t i = 0; i < n_states; ++i)
    if (rcs[i] != CK_OK) {
      first = rcs[i];
      break;
    }
  return first;
}

int ck_turn_noalloc(ck_model* m, void* dev_state, size_t len, void* stream, ck_turn_result* out) {
  if (!m || !dev_state || !out) return CK_INVALID_ARGUMENT;
  memset(out, 0, sizeof(*out));
  out->token = 0xFFFFFFFFu;
  if (reinterpret_cast<uintptr_t>(dev_state) % 256) return CK_INVALID_STATE;
  cudaStream_t s = S(stream);
  HostHeader h0;
  int rc = read_header(dev_state, &h0, s);
  if (rc) return rc;
  StateLayout lay;
  rc = check_state(m, dev_state, len, h0, &lay);
  if (rc) return rc;
  if (h0.u32(kHPhase) != CK_PHASE_RUNNING) return CK_INVALID_STATE;
  const uint32_t pos0 = h0.u32(kHPosition), np = h0.u32(kHNPrompt);
  if (pos0 >= lay.cache) return CK_INVALID_STATE;
  StepParams p;
  int grid;
  size_t smem;
  if (!plan_step(m, lay, &p, &grid, &smem, false)) return CK_INVALID_ARGUMENT;
  // scratch this position needs: counters, attention partials and accumulators, per-block
  // candidates, global planes
  const size_t need = step_work_bytes(p);
  if (need > noalloc_work_bytes()) return CK_INVALID_ARGUMENT;
  uint8_t* work = nullptr;
  CK_CUDA(noalloc_setup(m->step_smem, &work));
  p.st = static_cast<uint8_t*>(dev_state);
  p.generating = pos0 + 1 >= np ? 1u : 0u;
  CK_CUDA(cudaMemsetAsync(work, 0, p.zero_bytes, s));  // counters and sums start at zero every call
  CK_CUDA(launch_step_noalloc(p, work, s, grid, smem));
  HostHeader h1;
  rc = read_header(dev_state, &h1, s);
  if (rc) return rc;
  const bool failed = h1.u32(kHPhase) == CK_PHASE_FAILED;
  uint64_t turns = h1.u64(kHTurns) + 1;
  CK_CUDA(cudaMemcpyAsync(static_cast<uint8_t*>(dev_state) + kHTurns, &turns, 8,
                          cudaMemcpyHostToDevice, s));
  CK_CUDA(cudaStreamSynchronize(s));
  out->generated = h1.u32(kHGenerated);
  out->generated_this_turn = out->generated - h0.u32(kHGenerated);
  if (out->generated_this_turn) out->token = h1.u32(kHLastTok);
  out->work = h1.u32(kHPosition) - pos0 + (failed ? 1u : 0u);
  out->complete = h1.u32(kHPhase) != CK_PHASE_RUNNING;
  const uint64_t key = h1.u64(kHErrKey);
  if (key != kNoError) {
    out->err_position = (uint32_t)(key >> 44);
    out->err_layer = (uint32_t)(key >> 32) & 0xFFFu;
    out->err_phase = (uint32_t)(key >> 24) & 0xFFu;
    out->err_element = (uint32_t)key & 0xFFFFFFu;
  }
  return failed ? (int)h1.u32(kHError) : CK_OK;
}

int ck_logits(const ck_model* m, const void* dev_state, size_t len, int64_t* host_out, void* stream) {
  if (!m || !dev_state || !host_out) return CK_INVALID_ARGUMENT;
  cudaStream_t s = S(stream);
  HostHeader h;
  int rc = read_header(dev_state, &h, s);
  if (rc) return rc;
  StateLayout lay;
  rc = check_state(m, dev_state, len, h, &lay);
  if (rc) return rc;
  CK_CUDA(cudaMemcpyAsync(host_out, static_cast<const uint8_t*>(dev_state) + lay.logits,
                          8ull * m->cfg.vocab, cudaMemcpyDeviceToHost, s));
  CK_CUDA(cudaStreamSynchronize(s));
  return CK_OK;
}

int ck_argmax(const ck_model* m, const void* dev_state, size_t len, uint32_t* out, void* stream) {
  if (!m || !dev_state || !out) return CK_INVALID_ARGUMENT;
  cudaStream_t s = S(stream);
  HostHeader h;
  int rc = read_header(dev_state, &h, s);
  if (rc) return rc;
  StateLayout lay;
  rc = check_state(m, dev_state, len, h, &lay);
  if (rc) return rc;
  k_argmax<<<1, kArgThreads, 0, s>>>(
      reinterpret_cast<const int64_t*>(static_cast<const uint8_t*>(dev_state) + lay.logits),
      m->cfg.vocab, m->scratch);
  CK_CUDA(cudaGetLastError());
  CK_CUDA(cudaMemcpyAsync(out, m->scratch, 4, cudaMemcpyDeviceToHost, s));
  CK_CUDA(cudaStreamSynchronize(s));
  return CK_OK;
}

int ck_output_tokens(const ck_model* m, const void* dev_state, size_t len, uint32_t* host_out,
                     uint32_t cap, uint32_t* n, void* stream) {
  if (!m || !dev_state || !n || (cap && !host_out)) return CK_INVALID_ARGUMENT;
  cudaStream_t s = S(stream);
  HostHeader h;
  int rc = read_header(dev_state, &h, s);
  if (rc) return rc;
  StateLayout lay;
  rc = check_state(m, dev_state, len, h, &lay);
  if (rc) return rc;
  uint32_t g = h.u32(kHGenerated);
  if (g > cap) g = cap;
  if (g) {
    CK_CUDA(cudaMemcpyAsync(host_out, static_cast<const uint8_t*>(dev_state) + lay.out, 4ull * g,
                            cudaMemcpyDeviceToHost, s));
    CK_CUDA(cudaStreamSynchronize(s));
  }
  *n = g;
  return CK_OK;
}

int ck_state_download(const void* dev_state, size_t len, void* host, void* stream) {
  if (!dev_state || !host) return CK_INVALID_ARGUMENT;
  CK_CUDA(cudaMemcpyAsync(host, dev_state, len, cudaMemcpyDeviceToHost, S(stream)));
  CK_CUDA(cudaStreamSynchronize(S(stream)));
  return CK_OK;
}

int ck_state_upload(void* dev_state, const void* host, size_t len, void* stream) {
  if (!dev_state || !host) return CK_INVALID_ARGUMENT;
  CK_CUDA(cudaMemcpyAsync(dev_state, host, len, cudaMemcpyHostToDevice, S(stream)));
  CK_CUDA(cudaStreamSynchronize(S(stream)));
  return CK_OK;
}

int ck_matrow(const uint8_t* dev_W, size_t pitch, const uint32_t* dev_scale, uint32_t rows,
              uint32_t cols, const int64_t* dev_x, int64_t* dev_y, void* stream) {
  if (!dev_W || !dev_scale || !dev_x || !dev_y) return CK_INVALID_ARGUMENT;
  if (pitch % 16 || pitch > 16384 || cols < 1 || cols > pitch || rows < 1 || rows > (1u << 24))
    return CK_INVALID_ARGUMENT;
  if (reinterpret_cast<uintptr_t>(dev_W) % 16 || reinterpret_cast<uintptr_t>(dev_x) % 8 ||
      reinterpret_cast<uintptr_t>(dev_y) % 8 || reinterpret_cast<uintptr_t>(dev_scale) % 4)
    return CK_INVALID_ARGUMENT;
  int dev = 0, sms = 0;
  CK_CUDA(configure_matrow());
  CK_CUDA(cudaGetDevice(&dev));
  CK_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  MatrowParams p = {};
  p.W = dev_W;
  p.scale = dev_scale;
  p.grouped = 0;
  p.pitch = (uint32_t)pitch;
  p.rows = rows;
  p.cols = cols;
  p.pro = kProPlain;
  p.in = dev_x;
  p.epi = kEpiStore;
  p.out = dev_y;
  CK_CUDA(launch_matrow(p, S(stream), sms));
  return CK_OK;
}

}  // extern "C"
