// One position of the forward pass ("The inference core", "The forward pass, in order") as
// one persistent kernel: one CTA per SM, launched cooperatively so every CTA is resident.
//
// GB300 design.  Each CTA owns a contiguous slice of the rows of every matrix of the step,
// cut into panels of at most 96 rows.  The model's matrices sit in HBM in column-group
// layout (rows of 128-byte groups), so one panel's rows of one column group are a single
// contiguous run: a producer warp streams them, panel after panel, matrix after matrix and
// layer after layer, through a ring of shared-memory slots with cp.async.bulk copies that
// complete on mbarriers.  It never waits for activations, only for free slots, so HBM keeps
// streaming across phase boundaries.
//
// Eight consumer warps read every slot: warp w takes the 16-byte column chunk w of each
// column group, and lane l accumulates rows l, l + 32, ... of the panel, so a lane holds
// whole dot products over its columns and no shuffle reduction is needed: at the end of a
// panel the warps' partial sums meet in shared memory and one thread per row runs the
// fused epilogue.  The dot products use byte planes of the input vector: the phase's prologue
// (residual, RMS normalization) writes plane k = byte k of every element, and each row sum
// is sum_k 2^(8k) sum_c byte[r][c] * plane_k[c], one dp4a per four bytes and limb.
//
// Phases that depend on each other are separated by a grid barrier among the consumer
// warps.  Attention splits each head's positions over a few CTAs that add their weighted
// values into 64-bit accumulators in the work area; the CTAs of a head exchange maxima and
// sums only when the context is long enough to split the scoring.  Every wait is bounded:
// on a timeout the kernel raises an abort flag, stops issuing copies, waits (bounded) for
// its copies in flight and the state is marked failed with error 9.
#include <climits>

#include "ck_internal.cuh"

namespace ck {
namespace {

constexpr int kNCW = (int)kStepWarps;   // consumer warps
constexpr int kCT = 32 * kNCW;          // consumer threads
constexpr int kThreads = kCT + 32;      // plus one producer warp
constexpr uint32_t kPollLimit = 1u << 22;
constexpr int kRMax = (int)(kPanelRows / 32);  // rows a lane accumulates
constexpr uint32_t kBlockElems = 16u * kCT;     // prologue: 16 consecutive elements a thread

// work area offsets (bytes from the start of the state's scores/work region); [0, 4096) is
// zeroed before every launch
constexpr uint32_t kWBar = 0, kWAbort = 4, kWHeads = 64;

enum Pro : int { kPPlain = 0, kPNorm = 1, kPEmbedNorm = 2, kPAcc = 3 };
enum Epi : int { kEStore = 0, kEQKV = 1, kESiLU = 2, kELogits = 3 };
enum Kind : int { kQKV = 0, kATT = 1, kO = 2, kGU = 3, kDOWN = 4, kCLS = 5, kEND = 6 };

struct MR {
  const uint8_t* W;  // column-group layout
  const uint32_t* scale;
  uint32_t pitch, rows, cols;
  int pro;
  const int64_t* in;
  const int64_t* add;
  int64_t* res_out;
  const int32_t* norm_w;
  int epi;
  int64_t* out;
  int32_t* kc;
  int32_t* vc;
};

struct Shared {
  unsigned long long ra[kNCW], rbuf[kNCW];
  long long am_v[kNCW];
  uint32_t am_i[kNCW];
  unsigned long long S, orv;
  int abort;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"r"(kCT) : "memory"); }

// Dynamic shared memory: the ring (ns slots), the X region (byte planes, row scales and
// rotary row; attention reuses it), the partial row sums [kNCW][kPanelRows] and the ring's
// full and empty mbarriers.  Everything below is addressed from the kernel's parameter
// block and this symbol, so the compiler can re-derive addresses instead of keeping them
// live across phases.
extern __shared__ __align__(128) uint8_t smem[];

__device__ __forceinline__ uint8_t* ring_of() { return smem; }
__device__ __forceinline__ uint8_t* xreg(const StepParams& p) { return smem + (size_t)p.ns * kStageBytes; }
__device__ __forceinline__ unsigned long long* red_of(const StepParams& p) {
  return reinterpret_cast<unsigned long long*>(xreg(p) + p.x_bytes);
}
__device__ __forceinline__ uint64_t* full_of(const StepParams& p) {
  return reinterpret_cast<uint64_t*>(red_of(p) + kNCW * kPanelRows);
}
__device__ __forceinline__ uint64_t* empty_of(const StepParams& p) { return full_of(p) + p.ns; }

// The position's own values: the scratch area (the state's work region, or the
// allocation-free variant's array), the position and its token.
struct Pos {
  uint8_t* work;
  uint32_t pos, tok;
};
__device__ __forceinline__ uint32_t* gbar_of(const Pos& q) { return reinterpret_cast<uint32_t*>(q.work + kWBar); }
__device__ __forceinline__ uint32_t* gabort_of(const Pos& q) { return reinterpret_cast<uint32_t*>(q.work + kWAbort); }

__device__ __forceinline__ int64_t* st64(const StepParams& p, uint64_t off) {
  return reinterpret_cast<int64_t*>(p.st + off);
}

// The matrix-row phase of kind `k` in layer l:
//   QKV   attention norm of x (+ y of the previous layer, the sum kept in x), Q/K/V rows,
//         rotary on Q and K, checked cache stores of K and V
//   O     the head outputs (accumulators >> 24) times Wo, into y
//   GU    feed-forward norm of x + y (the sum kept in xb), gate and up rows, SiLU gating, h
//   DOWN  h times W2, into y
//   CLS   final norm of xb + y (the sum kept in x), the classifier rows into the logits
__device__ __forceinline__ MR matrow_of(const StepParams& p, const Pos& q, uint32_t l, int k) {
  MR m = {};
  const DevLayer* W = p.layers_tab + l;
  int64_t* x = st64(p, p.off_x);
  int64_t* xb = st64(p, p.off_xb);
  int64_t* y = st64(p, p.off_y);
  if (k == kQKV) {
    m.W = W->wqkv; m.scale = W->sqkv; m.pitch = p.pitch_d; m.rows = p.dim + 2 * p.kv_dim; m.cols = p.dim;
    m.pro = l == 0 ? kPEmbedNorm : kPNorm;
    m.in = xb; m.add = l == 0 ? nullptr : y; m.res_out = x; m.norm_w = W->attn_norm;
    m.epi = kEQKV; m.out = st64(p, p.off_q);
    const size_t lw = (size_t)p.cache * p.kv_dim;
    m.kc = reinterpret_cast<int32_t*>(p.st + p.off_k) + l * lw;
    m.vc = reinterpret_cast<int32_t*>(p.st + p.off_v) + l * lw;
  } else if (k == kO) {
    m.W = W->wo; m.scale = W->so; m.pitch = p.pitch_d; m.rows = p.dim; m.cols = p.dim;
    m.pro = kPAcc; m.in = reinterpret_cast<const int64_t*>(q.work + p.off_oacc); m.epi = kEStore; m.out = y;
  } else if (k == kGU) {
    m.W = W->w13; m.scale = W->s13; m.pitch = p.pitch_d; m.rows = 2 * p.hidden; m.cols = p.dim;
    m.pro = kPNorm; m.in = x; m.add = y; m.res_out = xb; m.norm_w = W->ffn_norm;
    m.epi = kESiLU; m.out = st64(p, p.off_h);
  } else if (k == kDOWN) {
    m.W = W->w2; m.scale = W->s2; m.pitch = p.pitch_h; m.rows = p.dim; m.cols = p.hidden;
    m.pro = kPPlain; m.in = st64(p, p.off_h); m.epi = kEStore; m.out = y;
  } else {  // classifier
    m.W = p.cls; m.scale = p.cls_scale; m.pitch = p.pitch_d; m.rows = p.vocab; m.cols = p.dim;
    m.pro = kPNorm; m.in = xb; m.add = y; m.res_out = x; m.norm_w = p.final_norm;
    m.epi = kELogits; m.out = st64(p, p.off_logits);
  }
  return m;
}

// This CTA's rows of a matrix: whole pairs, split evenly over the grid.
__device__ __forceinline__ void cta_rows(uint32_t rows, uint32_t b, uint32_t G, uint32_t& rb, uint32_t& re) {
  const uint32_t np = (rows + 1) / 2;
  const uint32_t pb = (uint32_t)((uint64_t)np * b / G), pe = (uint32_t)((uint64_t)np * (b + 1) / G);
  rb = min(rows, 2 * pb);
  re = min(rows, 2 * pe);
}
__device__ __forceinline__ uint32_t panel_count(uint32_t nr) { return (nr + kPanelRows - 1) / kPanelRows; }
// Panel i of npan over nr rows: rows [p0, p0 + pn) of the CTA's slice, whole pairs, at most
// kPanelRows (ceil(nr / 2) <= (kPanelRows / 2) npan pairs, split evenly).
__device__ __forceinline__ void panel_of(uint32_t nr, uint32_t npan, uint32_t i, uint32_t& p0, uint32_t& pn) {
  const uint32_t pairs = (nr + 1) / 2;
  const uint32_t a = pairs * i / npan, b = pairs * (i + 1) / npan;
  p0 = 2 * a;
  pn = min(2 * b, nr) - 2 * a;
}
// Column groups one ring slot holds for a panel of pn rows (at least one: pn * 128 <= slot).
__device__ __forceinline__ uint32_t groups_per_stage(uint32_t pn) {
  const uint32_t g = kStageBytes / (pn * kGroupCols);
  return g < 1 ? 1 : g;
}

// ------------------------------------------------------------------ producer

__device__ bool producer_wait_empty(const StepParams& p, const Pos& q, uint32_t slot, uint32_t parity) {
  for (uint32_t i = 0; i < kPollLimit; ++i) {
    if (mbar_try(&empty_of(p)[slot], parity)) return true;
    if ((i & 63) == 63 && ld_acquire(gabort_of(q))) return false;
  }
  atomicExch(gabort_of(q), 1u);
  return false;
}

__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Walks the position's ring stages in order: layer, matrix, panel, column groups.  Stage =
// ng runs of `run` bytes, run r starting at src + r * gstride.
struct StageCursor {
  uint32_t l, kk;        // layer and matrix index (QKV, O, GU, DOWN; the classifier after)
  uint32_t rb, nr, npan, pi, p0, pn, gps, g0, NG;
  const uint8_t* W;
  uint32_t rows;
  bool done;
};

// The matrix of (l, kk), or false past the last one.
__device__ __forceinline__ bool cursor_matrix(const StepParams& p, const Pos& q, StageCursor& c) {
  for (;;) {
    if (c.l > p.layers || (c.l == p.layers && (!p.generating || c.kk > 0))) return false;
    int k = c.kk == 0 ? kQKV : c.kk == 1 ? kO : c.kk == 2 ? kGU : kDOWN;
    if (c.l == p.layers) k = kCLS;
    const MR m = matrow_of(p, q, c.l < p.layers ? c.l : 0, k);
    uint32_t re;
    cta_rows(m.rows, blockIdx.x, gridDim.x, c.rb, re);
    c.nr = re - c.rb;
    c.npan = panel_count(c.nr);
    c.NG = m.pitch / kGroupCols;
    c.W = m.W;
    c.rows = m.rows;
    c.pi = 0;
    c.g0 = 0;
    if (c.npan) {
      panel_of(c.nr, c.npan, 0, c.p0, c.pn);
      c.gps = groups_per_stage(c.pn);
      return true;
    }
    if (++c.kk == 4) {
      c.kk = 0;
      ++c.l;
    }
  }
}
__device__ __forceinline__ void cursor_start(const StepParams& p, const Pos& q, StageCursor& c) {
  c.l = 0;
  c.kk = 0;
  c.done = !cursor_matrix(p, q, c);
}
__device__ __forceinline__ void cursor_next(const StepParams& p, const Pos& q, StageCursor& c) {
  c.g0 += c.gps;
  if (c.g0 < c.NG) return;
  c.g0 = 0;
  if (++c.pi < c.npan) {
    panel_of(c.nr, c.npan, c.pi, c.p0, c.pn);
    c.gps = groups_per_stage(c.pn);
    return;
  }
  if (++c.kk == 4) {
    c.kk = 0;
    ++c.l;
  }
  c.done = !cursor_matrix(p, q, c);
}

// The producer: fills ring slot gs % ns with stage gs once the slot's previous stage is
// released, and keeps L2 prefetches of the following stages about pf_bytes ahead of the
// fills, so that HBM keeps streaming while the consumers are in barriers, prologues or
// attention and the ring is full.
__device__ void producer(const StepParams& p, const Pos& q) {
  uint64_t* full = full_of(p);
  const uint32_t ns = p.ns;
  StageCursor fc, pc;
  cursor_start(p, q, fc);
  cursor_start(p, q, pc);
  unsigned long long filled = 0, fetched = 0;  // bytes
  uint32_t gs = 0;
  bool ok = true;
  for (; !fc.done; cursor_next(p, q, fc), ++gs) {
    const uint32_t run = fc.pn * kGroupCols;
    const uint32_t ng = min(fc.gps, fc.NG - fc.g0);
    // prefetch ahead (the fill cursor never passes the prefetch cursor)
    while (p.pf_bytes && !pc.done && fetched < filled + ng * run + p.pf_bytes) {
      const uint32_t prun = pc.pn * kGroupCols, png = min(pc.gps, pc.NG - pc.g0);
      const uint8_t* src = pc.W + (size_t)(pc.rb + pc.p0) * kGroupCols + (size_t)pc.g0 * pc.rows * kGroupCols;
      for (uint32_t gl = 0; gl < png; ++gl) prefetch_l2(src + (size_t)gl * pc.rows * kGroupCols, prun);
      fetched += (unsigned long long)png * prun;
      cursor_next(p, q, pc);
    }
    const uint32_t slot = gs % ns;
    if (gs >= ns && !producer_wait_empty(p, q, slot, ((gs / ns) - 1) & 1)) {
      ok = false;
      break;
    }
    if (gs >= ns && !mbar_try(&full[slot], ((gs / ns) - 1) & 1)) {
      atomicExch(gabort_of(q), 1u);  // the slot's last fill never completed: stop, do not re-arm
      ok = false;
      break;
    }
    mbar_expect_tx(&full[slot], ng * run);
    uint8_t* dst = ring_of() + (size_t)slot * kStageBytes;
    const uint8_t* src = fc.W + (size_t)(fc.rb + fc.p0) * kGroupCols + (size_t)fc.g0 * fc.rows * kGroupCols;
    for (uint32_t gl = 0; gl < ng; ++gl)
      bulk_g2s(dst + (size_t)gl * run, src + (size_t)gl * fc.rows * kGroupCols, run, &full[slot]);
    filled += (unsigned long long)ng * run;
  }
  (void)ok;
  // wait (bounded) for every copy still in flight before the CTA may exit
  for (uint32_t j = gs > ns ? gs - ns : 0; j < gs; ++j) {
    for (uint32_t i = 0; i < kPollLimit; ++i)
      if (mbar_try(&full[j % ns], (j / ns) & 1)) break;
  }
}

// ------------------------------------------------------------------ consumer helpers

// Barrier over the consumer warps of every CTA; `epoch` counts the barriers passed.  The
// release add publishes this CTA's writes (ordered before it by the CTA barrier), and the
// acquire load that sees every CTA's add orders the others' writes before this CTA's reads.
__device__ bool grid_sync(const Pos& q, Shared& sh, uint32_t& epoch) {
  consumer_bar();
  ++epoch;
  if (threadIdx.x == 0) {
    uint32_t* gbar = gbar_of(q);
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(gbar) : "memory");
    const uint32_t target = epoch * gridDim.x;
    uint32_t i = 0;
    while (ld_acquire(gbar) < target) {
      if (++i > kPollLimit || ((i & 255) == 0 && ld_acquire(gabort_of(q)))) {
        atomicExch(gabort_of(q), 1u);
        sh.abort = 1;
        break;
      }
    }
  }
  consumer_bar();
  return sh.abort == 0;
}

// Barrier among the gh CTAs of one attention head (monotonic target within a launch).
__device__ bool group_sync(const Pos& q, Shared& sh, uint32_t* counter, uint32_t target) {
  consumer_bar();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
    uint32_t i = 0;
    while (ld_acquire(counter) < target) {
      if (++i > kPollLimit || ((i & 255) == 0 && ld_acquire(gabort_of(q)))) {
        atomicExch(gabort_of(q), 1u);
        sh.abort = 1;
        break;
      }
    }
  }
  consumer_bar();
  return sh.abort == 0;
}

__device__ __forceinline__ unsigned long long warp_sum(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ unsigned long long warp_or(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum and OR over the consumer threads (all get the results).
__device__ void consumer_sum_or(unsigned long long& s, unsigned long long& o, Shared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  s = warp_sum(s);
  o = warp_or(o);
  if (lane == 0) {
    sh.ra[warp] = s;
    sh.rbuf[warp] = o;
  }
  consumer_bar();
  unsigned long long a = 0, b = 0;
#pragma unroll
  for (int w = 0; w < kNCW; ++w) {
    a += sh.ra[w];
    b |= sh.rbuf[w];
  }
  consumer_bar();  // every thread has read the partials before they are reused
  s = a;
  o = b;
}

// The phase input for elements e0 .. e0+15 (e0 a multiple of 16): the embedding row of the
// token (phase 3), the attention accumulators >> 24, or in (+ add).  Zeros at and beyond n.
__device__ __forceinline__ void load16(const StepParams& p, const Pos& q, const MR& m, uint32_t e0,
                                       int64_t (&x)[16]) {
  const uint32_t n = m.cols;
  if (m.pro == kPEmbedNorm) {
    const int64_t s = (int64_t)__ldg(p.embed_scale + q.tok);
    uint4 b = make_uint4(0u, 0u, 0u, 0u);
    if (e0 < n) b = __ldg(reinterpret_cast<const uint4*>(p.embed + grouped_offset(p.vocab, q.tok, e0)));
    const uint32_t wd[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int64_t byte = (int64_t)((wd[i >> 2] >> (8 * (i & 3))) & 0xFFu);
      x[i] = e0 + i < n ? (byte - 128) * s >> 8 : 0;
    }
    return;
  }
  if (e0 + 16 <= n) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const longlong2 v = *reinterpret_cast<const longlong2*>(m.in + e0 + 2 * j);
      x[2 * j] = v.x;
      x[2 * j + 1] = v.y;
    }
    if (m.add) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const longlong2 v = *reinterpret_cast<const longlong2*>(m.add + e0 + 2 * j);
        x[2 * j] = wadd(x[2 * j], v.x);
        x[2 * j + 1] = wadd(x[2 * j + 1], v.y);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      int64_t v = 0;
      if (e0 + i < n) {
        v = m.in[e0 + i];
        if (m.add) v = wadd(v, m.add[e0 + i]);
      }
      x[i] = v;
    }
  }
  if (m.pro == kPAcc) {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] >>= 24;
  }
}

// The norm weights of elements e0 .. e0+15 (zeros beyond n).
__device__ __forceinline__ void load_w16(const MR& m, uint32_t e0, int32_t (&w)[16]) {
  const uint32_t n = m.cols;
  if (e0 + 16 <= n) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int4 v = __ldg(reinterpret_cast<const int4*>(m.norm_w + e0 + 4 * j));
      w[4 * j] = v.x;
      w[4 * j + 1] = v.y;
      w[4 * j + 2] = v.z;
      w[4 * j + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = e0 + i < n ? __ldg(m.norm_w + e0 + i) : 0;
  }
}

// Planes k0 .. k1-1 of the 16 values: plane k's bytes (byte k of each value, in element
// order) are 16 bytes at base + (k - kbase) * pitch + e0.  A 4 x 4 byte transpose of each
// group of four values gives their four low (or high) plane words.
__device__ __forceinline__ void store_planes(const int64_t (&y)[16], uint8_t* base, uint32_t pitch,
                                             uint32_t e0, uint32_t k0, uint32_t k1, uint32_t kbase) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    if ((uint32_t)(4 * half) >= k1 || (uint32_t)(4 * half + 4) <= k0) continue;
    uint32_t pw[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t a = (uint32_t)((uint64_t)y[4 * q] >> (32 * half));
      const uint32_t b = (uint32_t)((uint64_t)y[4 * q + 1] >> (32 * half));
      const uint32_t cc = (uint32_t)((uint64_t)y[4 * q + 2] >> (32 * half));
      const uint32_t d = (uint32_t)((uint64_t)y[4 * q + 3] >> (32 * half));
      const uint32_t ab0 = __byte_perm(a, b, 0x5140), ab1 = __byte_perm(a, b, 0x7362);
      const uint32_t cd0 = __byte_perm(cc, d, 0x5140), cd1 = __byte_perm(cc, d, 0x7362);
      pw[0][q] = __byte_perm(ab0, cd0, 0x5410);
      pw[1][q] = __byte_perm(ab0, cd0, 0x7632);
      pw[2][q] = __byte_perm(ab1, cd1, 0x5410);
      pw[3][q] = __byte_perm(ab1, cd1, 0x7632);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t k = 4 * half + j;
      if (k < k0 || k >= k1) continue;
      *reinterpret_cast<uint4*>(base + (size_t)(k - kbase) * pitch + e0) =
          make_uint4(pw[j][0], pw[j][1], pw[j][2], pw[j][3]);
    }
  }
}

// Packs the phase's input vector into byte planes (after the residual and the RMS
// normalization where the phase has them): planes below *lcap_out in shared memory, the
// others (only when the vector needs them) in the global copy.  Returns the limb count and
// *S_out the wrapping sum of the packed vector.  Also stages this CTA's row scales and (for
// Q/K/V) the position's rotary row in shared memory, and for Q/K/V block 0 clears the
// attention accumulators that this layer's attention adds into.
__device__ __forceinline__ int prologue(const StepParams& p, const Pos& q, const MR& m, Shared& sh,
                                        unsigned long long* S_out, uint32_t* lcap_out) {
  const uint32_t n = m.cols, pitch = m.pitch;
  uint8_t* X = xreg(p);
  const uint32_t nblk = (pitch + kBlockElems - 1) / kBlockElems;
  uint32_t lcap = p.planes_bytes / pitch;
  if (lcap > 8) lcap = 8;
  const bool writer = blockIdx.x == 0;
  const bool norm = m.pro == kPNorm || m.pro == kPEmbedNorm;
  const uint32_t tid = threadIdx.x, et = 16 * tid;
  uint32_t rb, re;
  cta_rows(m.rows, blockIdx.x, gridDim.x, rb, re);
  uint32_t* sc = reinterpret_cast<uint32_t*>(X + p.planes_bytes);
  int32_t* rp = reinterpret_cast<int32_t*>(X + p.planes_bytes + 4 * p.scale_cap);
  const bool qkv = m.epi == kEQKV;
  // loads whose results are only stored at the end: in flight during the vector work
  const uint32_t my_row = rb + tid;
  const uint32_t my_scale = my_row < re ? __ldg(m.scale + my_row) : 0u;
  const int32_t my_rope = (qkv && tid < p.hd) ? __ldg(p.rope + (size_t)q.pos * p.hd + tid) : 0;
  if (qkv && writer) {
    unsigned long long* acc = reinterpret_cast<unsigned long long*>(q.work + p.off_oacc);
    for (uint32_t i = tid; i < p.dim; i += kCT) acc[i] = 0ull;
  }
  int64_t x[16];
  int32_t w[16];
  InvDiv D = {};
  if (norm) {
    // "RMS normalization": rms = isqrt(sum(x*x)/n + 42,950), at least 1
    unsigned long long ss = 0, dummy = 0;
    for (uint32_t b = 0; b < nblk; ++b) {
      const uint32_t e0 = b * kBlockElems + et;
      if (e0 >= pitch) continue;
      load16(p, q, m, e0, x);
      if (nblk == 1) load_w16(m, e0, w);  // in flight while the sums reduce
#pragma unroll
      for (int i = 0; i < 16; ++i) ss += (unsigned long long)x[i] * (unsigned long long)x[i];
      if (writer && m.res_out) {
        if (e0 + 16 <= n) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            longlong2 v;
            v.x = x[2 * j];
            v.y = x[2 * j + 1];
            *reinterpret_cast<longlong2*>(m.res_out + e0 + 2 * j) = v;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (e0 + i < n) m.res_out[e0 + i] = x[i];
        }
      }
    }
    consumer_sum_or(ss, dummy, sh);
    const InvDiv& Dn = n == p.dim ? p.div_dim : p.div_hidden;
    uint64_t rms = isqrt_u64(udiv_inv(ss, Dn) + 42950ull);
    if (rms < 1) rms = 1;
    D = make_invdiv((uint32_t)rms);  // every thread alike: no broadcast needed
  }
  unsigned long long S = 0, orv = 0;
  for (uint32_t b = 0; b < nblk; ++b) {
    const uint32_t e0 = b * kBlockElems + et;
    if (e0 >= pitch) continue;
    if (!(norm && nblk == 1)) {  // a single block is still in registers
      load16(p, q, m, e0, x);
      if (norm) load_w16(m, e0, w);
    }
    if (norm) {
      // y = ((x * w) / rms) >> 8, the division truncating toward zero (zeros beyond n)
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = sdiv_trunc(wmul(x[i], (int64_t)w[i]), D) >> 8;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      S += (unsigned long long)x[i];
      orv |= (unsigned long long)(x[i] ^ (x[i] >> 63));
    }
    store_planes(x, X, pitch, e0, 0, lcap, 0);
  }
  if (my_row < re) sc[tid] = my_scale;
  for (uint32_t r = my_row + kCT; r < re; r += kCT) sc[r - rb] = __ldg(m.scale + r);
  if (qkv && tid < p.hd) rp[tid] = my_rope;
  for (uint32_t i = tid + kCT; qkv && i < p.hd; i += kCT) rp[i] = __ldg(p.rope + (size_t)q.pos * p.hd + i);
  consumer_sum_or(S, orv, sh);  // its barriers also publish the planes, scales and rotary row
  int L = 1;
  while (L < 8 && (orv >> (8 * L - 1)) != 0) ++L;
  if (L > 4) L = 8;  // the consumers run 1, 2, 3, 4 or 8 limbs
  if ((uint32_t)L > lcap) {
    // A vector beyond 8*lcap bits (rare): its planes lcap..L-1 go to the global copy, which
    // every block writes with the same bytes after the grid barrier that opened the phase.
    uint8_t* gpl = q.work + p.off_gplanes;
    for (uint32_t b = 0; b < nblk; ++b) {
      const uint32_t e0 = b * kBlockElems + et;
      if (e0 >= pitch) continue;
      if (nblk > 1) {  // one block is still in registers
        load16(p, q, m, e0, x);
        if (norm) {
          load_w16(m, e0, w);
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = sdiv_trunc(wmul(x[i], (int64_t)w[i]), D) >> 8;
        }
      }
      store_planes(x, gpl, pitch, e0, lcap, (uint32_t)L, lcap);
    }
    __threadfence_block();
    consumer_bar();
  }
  *S_out = S;
  *lcap_out = lcap;
  return L;
}

// ------------------------------------------------------------------ matrix rows

struct Best {
  long long v;
  uint32_t i;
};

__device__ __forceinline__ void best_update(Best& b, long long v, uint32_t i) {
  if (b.i == 0xFFFFFFFFu || v > b.v || (v == b.v && i < b.i)) {
    b.v = v;
    b.i = i;
  }
}

// Epilogue of one row (threads with valid == false only take part in the partner exchange;
// the partner of an even row is the next thread).
__device__ __forceinline__ void epilogue(const StepParams& p, const Pos& q, const MR& m, uint32_t layer,
                                         uint32_t row, bool valid, int64_t y, Best& best, const int32_t* rope) {
  const int64_t partner = (int64_t)__shfl_xor_sync(0xffffffffu, (unsigned long long)y, 1);
  if (!valid) return;
  if (m.epi == kEStore) {
    m.out[row] = y;
  } else if (m.epi == kELogits) {
    m.out[row] = y;
    best_update(best, y, row);
  } else if (m.epi == kESiLU) {
    if ((row & 1) == 0) m.out[row >> 1] = wmul(silu_lookup(y, p.silu_tab), partner) >> 16;
  } else {  // Q/K/V: rotary on Q and K, checked cache stores for K and V
    const bool even = (row & 1) == 0;
    const int64_t a = even ? y : partner, b = even ? partner : y;
    const uint32_t q_rows = p.dim;
    if (row < q_rows) {
      const uint32_t j = (row % p.hd) >> 1;
      int64_t a2, b2;
      rotate_pair(a, b, rope[2 * j], rope[2 * j + 1], a2, b2);
      m.out[row] = even ? a2 : b2;
    } else if (row < q_rows + p.kv_dim) {
      const uint32_t e = row - q_rows;
      if (!fits_i32(y)) record_error(p.st, err_key(q.pos, layer, 6, e));
      const uint32_t j = (e % p.hd) >> 1;
      int64_t a2, b2;
      rotate_pair((int64_t)(int32_t)a, (int64_t)(int32_t)b, rope[2 * j], rope[2 * j + 1], a2, b2);
      const int64_t mine = even ? a2 : b2;
      if (!fits_i32(mine)) record_error(p.st, err_key(q.pos, layer, 8, e));
      m.kc[(size_t)q.pos * p.kv_dim + e] = (int32_t)mine;
    } else {
      const uint32_t e = row - q_rows - p.kv_dim;
      if (!fits_i32(y)) record_error(p.st, err_key(q.pos, layer, 7, e));
      m.vc[(size_t)q.pos * p.kv_dim + e] = (int32_t)y;
    }
  }
}

// Waits (bounded) for a ring slot's fill; false after a timeout or another CTA's abort.
__device__ __forceinline__ bool wait_full(const StepParams& p, const Pos& q, uint32_t slot, uint32_t parity) {
  for (uint32_t i = 0; i < kPollLimit; ++i) {
    if (mbar_try(&full_of(p)[slot], parity)) return true;
    if ((i & 63) == 63 && ld_acquire(gabort_of(q))) return false;
  }
  atomicExch(gabort_of(q), 1u);
  return false;
}

// dp4a of one weight chunk (16 bytes of a row) with one plane chunk into a limb sum: plain
// u8 x u8 for the low planes, u8 x s8 for the top plane (top is a constant after
// unrolling).
__device__ __forceinline__ uint32_t dp16(bool top, const uint4& w, const uint4& x, uint32_t a) {
  if (top) {
    int t = dp4a_us(w.x, x.x, (int)a);
    t = dp4a_us(w.y, x.y, t);
    t = dp4a_us(w.z, x.z, t);
    t = dp4a_us(w.w, x.w, t);
    return (uint32_t)t;
  }
  a = __dp4a(w.x, x.x, a);
  a = __dp4a(w.y, x.y, a);
  a = __dp4a(w.z, x.z, a);
  return __dp4a(w.w, x.w, a);
}

// This warp's share of one ring stage (ng column groups of a panel) for R row slots and
// L <= 4 limbs: lane = row slot (rows lane + 32 j of the panel), warp = 16-byte column
// chunk of every group; acc[j][k] is the u32 sum of row slot j's bytes times plane k (the
// top plane L-1 signed; all in shared memory, which holds at least four).  `pc` is the
// lane's chunk position within a row's 128 bytes (the warp's chunk rotated by the rows'
// index in the matrix, modulo 8).  (One group at a time: with nine warps a thread has 168
// registers, and two groups in flight made the compiler spill.)
template <int R, int L>
__device__ __forceinline__ void stage_narrow(const uint8_t* stage, uint32_t ng, uint32_t run,
                                             const uint32_t (&roff)[kRMax], uint32_t pc, uint32_t col0,
                                             const uint8_t* planes, uint32_t pitch,
                                             uint32_t (&acc)[kRMax][4]) {
#pragma unroll 1
  for (uint32_t gl = 0; gl < ng; ++gl) {
    const uint8_t* base = stage + (size_t)gl * run + pc;
    const uint8_t* xcol = planes + col0 + gl * kGroupCols;
    uint4 wv[R];
#pragma unroll
    for (int j = 0; j < R; ++j) wv[j] = *reinterpret_cast<const uint4*>(base + roff[j]);
#pragma unroll
    for (int k = 0; k < L; ++k) {
      const uint4 xk = *reinterpret_cast<const uint4*>(xcol + (size_t)k * pitch);
#pragma unroll
      for (int j = 0; j < R; ++j) acc[j][k] = dp16(k == L - 1, wv[j], xk, acc[j][k]);
    }
  }
}

// The same for vectors of 5 to 8 limbs (rare): all eight planes (planes above the last are
// the sign bytes, so the sum with the top plane signed is still exact), each chunk's limb
// sums folded at once into a wrapping 64-bit sum per row slot kept in acc[j][0] (low word)
// and acc[j][1] (high word), so that no eight u32 accumulators per row stay live.  Planes
// k >= lcap come from the global copy.
template <int R>
__device__ __forceinline__ void stage_wide(const uint8_t* stage, uint32_t ng, uint32_t run,
                                           const uint32_t (&roff)[kRMax], uint32_t pc, uint32_t col0,
                                           const uint8_t* planes, const uint8_t* gpl, uint32_t pitch,
                                           uint32_t lcap, uint32_t (&acc)[kRMax][4]) {
#pragma unroll 1
  for (uint32_t gl = 0; gl < ng; ++gl) {
    const uint8_t* base = stage + (size_t)gl * run + pc;
    const uint32_t col = col0 + gl * kGroupCols;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const uint4 w = *reinterpret_cast<const uint4*>(base + roff[j]);
      unsigned long long sum = ((unsigned long long)acc[j][1] << 32) | acc[j][0];
#pragma unroll 1
      for (int k = 0; k < 8; ++k) {
        uint4 xk;
        if ((uint32_t)k < lcap) xk = *reinterpret_cast<const uint4*>(planes + (size_t)k * pitch + col);
        else xk = *reinterpret_cast<const uint4*>(gpl + (size_t)(k - lcap) * pitch + col);  // written in this launch
        if (k < 7) sum += (unsigned long long)dp16(false, w, xk, 0u) << (8 * k);
        else sum += (unsigned long long)(long long)(int)dp16(true, w, xk, 0u) << 56;
      }
      acc[j][0] = (uint32_t)sum;
      acc[j][1] = (uint32_t)(sum >> 32);
    }
  }
}

// The consumers' next ring stage: its slot and the parity of the fill it waits for.
struct RingPos {
  uint32_t slot, par;
};
__device__ __forceinline__ void ring_advance(const StepParams& p, RingPos& r) {
  if (++r.slot == p.ns) {
    r.slot = 0;
    r.par ^= 1u;
  }
}

// Waits for each stage of a panel (NG column groups, gps a stage), runs this warp's share
// with the body for (R row slots, L limbs) and releases the slot.  A warp that meets a
// timeout (or sees another's) keeps walking the stages without waiting, so that every warp
// reaches the same CTA barriers; returns whether it did.
template <int R, int L>
__device__ __forceinline__ bool panel_stages(const StepParams& p, const Pos& q, RingPos& rp, uint32_t NG,
                                             uint32_t gps, uint32_t run, const uint32_t (&roff)[kRMax],
                                             uint32_t pc, uint32_t col0, const uint8_t* planes,
                                             const uint8_t* gpl, uint32_t pitch, uint32_t lcap, Shared& sh,
                                             bool dead, uint32_t (&acc)[kRMax][4]) {
  const uint32_t lane = threadIdx.x & 31;
  for (uint32_t g0 = 0; g0 < NG; g0 += gps) {
    const uint32_t slot = rp.slot;
    if (!dead && *reinterpret_cast<volatile int*>(&sh.abort)) dead = true;
    if (!dead && !wait_full(p, q, slot, rp.par)) {
      dead = true;
      sh.abort = 1;
    }
    if (!dead) {
      const uint32_t ng = min(gps, NG - g0);
      const uint8_t* stage = ring_of() + (size_t)slot * kStageBytes;
      if (L <= 4) stage_narrow<R, (L <= 4 ? L : 4)>(stage, ng, run, roff, pc, col0 + g0 * kGroupCols, planes, pitch, acc);
      else stage_wide<R>(stage, ng, run, roff, pc, col0 + g0 * kGroupCols, planes, gpl, pitch, lcap, acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_of(p)[slot]);
    ring_advance(p, rp);
  }
  return dead;
}

// One matrix-row phase on this CTA's rows.  Every warp reads every stage (warp w: column
// chunk w of each group) and accumulates the rows in registers (lane = row), so all warps
// finish a panel together; at the end of each panel the warps' partial sums are added in
// shared memory and one thread per row applies the correction, the row scale and the
// epilogue: y = ((sum_c byte * x - 128 * S) * scale) >> 24, wrapping in 64 bits.  A warp that meets a timeout keeps walking the stages without waiting, so
// that every warp reaches the same CTA barriers; the caller leaves on sh.abort.
__device__ __forceinline__ void consume_phase(const StepParams& p, const Pos& q, const MR& m, uint32_t layer,
                                              int L, unsigned long long S, uint32_t lcap, RingPos& rp,
                                              Shared& sh, Best& best) {
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  uint32_t rb, re;
  cta_rows(m.rows, blockIdx.x, gridDim.x, rb, re);
  const uint32_t nr = re - rb, npan = panel_count(nr), NG = m.pitch / kGroupCols;
  const uint32_t pitch = m.pitch;
  const uint8_t* planes = xreg(p);
  const uint8_t* gpl = q.work + p.off_gplanes;
  const uint32_t* sc = reinterpret_cast<const uint32_t*>(xreg(p) + p.planes_bytes);
  const int32_t* rope = reinterpret_cast<const int32_t*>(xreg(p) + p.planes_bytes + 4 * p.scale_cap);
  unsigned long long* red = red_of(p);
  bool dead = false;
  for (uint32_t pi = 0; pi < npan; ++pi) {
    uint32_t p0, pn;
    panel_of(nr, npan, pi, p0, pn);
    const uint32_t R = (pn + 31) / 32, gps = groups_per_stage(pn), run = pn * kGroupCols;
    const uint32_t pc = (warp ^ ((rb + p0 + lane) & 7u)) << 4;
    uint32_t roff[kRMax];
#pragma unroll
    for (int j = 0; j < kRMax; ++j) roff[j] = min(lane + 32u * j, pn - 1) * kGroupCols;
    uint32_t acc[kRMax][4];
#pragma unroll
    for (int j = 0; j < kRMax; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[j][k] = 0;
    const uint32_t col0 = warp * 16;
#define CK_PANEL(r, l)                                                                              \
  case r * 16 + l:                                                                                  \
    dead = panel_stages<r, l>(p, q, rp, NG, gps, run, roff, pc, col0, planes, gpl, pitch, lcap, sh, \
                              dead, acc);                                                           \
    break;
#define CK_PANELS(r) CK_PANEL(r, 1) CK_PANEL(r, 2) CK_PANEL(r, 3) CK_PANEL(r, 4) CK_PANEL(r, 8)
    switch (R * 16 + (uint32_t)L) {
      CK_PANELS(1) CK_PANELS(2) CK_PANELS(3)
      default: break;
    }
#undef CK_PANELS
#undef CK_PANEL
    // this warp's partial sums of the panel's rows, limbs combined (zero without stages)
#pragma unroll
    for (int j = 0; j < kRMax; ++j) {
      const uint32_t r = lane + 32u * j;
      if ((uint32_t)j >= R || r >= pn) continue;
      unsigned long long a = 0;
      if (L <= 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (k >= L) continue;
          const unsigned long long t = (k < L - 1) ? (unsigned long long)acc[j][k]
                                                   : (unsigned long long)(long long)(int)acc[j][k];
          a += t << (8 * k);
        }
      } else {
        a = ((unsigned long long)acc[j][1] << 32) | acc[j][0];
      }
      red[warp * kPanelRows + r] = a;
    }
    consumer_bar();
    const bool valid = tid < pn && !dead;
    int64_t y = 0;
    if (valid) {
      unsigned long long sum = 0;
#pragma unroll
      for (int w = 0; w < kNCW; ++w) sum += red[w * kPanelRows + tid];
      const unsigned long long t = (sum - (S << 7)) * (unsigned long long)sc[p0 + tid];
      y = (int64_t)t >> 24;
    }
    epilogue(p, q, m, layer, rb + p0 + tid, valid, y, best, rope);
    consumer_bar();  // every thread has read the partial sums before the next panel's
  }
}

// ------------------------------------------------------------------ attention

// Phase 9 for this CTA's (head, chunk): "Attention" in four stages over positions 0..pos of
// the head's cache.  Each CTA adds sum_t P_t * v_t over its chunk of positions into the
// head's 64-bit accumulators (the O prologue applies the final >> 24).  The maximum and the
// sum Z need every position: for short contexts each CTA scores all positions itself; for
// longer ones the CTAs score their own chunks and exchange maxima and sums (two barriers
// among the head's CTAs).
__device__ __forceinline__ bool attention(const StepParams& p, const Pos& q, uint32_t l, Shared& sh) {
  const uint32_t b = blockIdx.x, gh = p.gh;
  if (b >= p.heads * gh) return true;
  const uint32_t h = b / gh, ch = b % gh, hd = p.hd;
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int64_t* q_s = reinterpret_cast<int64_t*>(xreg(p));
  unsigned long long* part = reinterpret_cast<unsigned long long*>(q_s + hd);  // [kNCW][hd]
  long long* red = reinterpret_cast<long long*>(part + kNCW * hd);             // [kNCW]
  long long* sc = red + kNCW;                                                  // scores
  const uint32_t P = q.pos + 1;
  const bool full = gh == 1 || P <= p.att_full;
  const uint32_t cs = (P + gh - 1) / gh;
  const uint32_t t0 = min(P, ch * cs), t1 = min(P, t0 + cs);
  const uint32_t s0 = full ? 0u : t0, s1 = full ? P : t1, nsc = s1 - s0;
  const uint32_t kvh = h / (p.heads / p.kv_heads);
  const size_t lw = (size_t)p.cache * p.kv_dim;
  const int32_t* Kh = reinterpret_cast<const int32_t*>(p.st + p.off_k) + l * lw + (size_t)kvh * hd;
  const int32_t* Vh = reinterpret_cast<const int32_t*>(p.st + p.off_v) + l * lw + (size_t)kvh * hd;
  long long* parts = reinterpret_cast<long long*>(q.work + p.off_part) + (size_t)h * gh * 2;  // [gh][2]
  uint32_t* hcount = reinterpret_cast<uint32_t*>(q.work + kWHeads) + h;
  const int64_t* qg = st64(p, p.off_q) + (size_t)h * hd;
  for (uint32_t i = tid; i < hd; i += kCT) q_s[i] = qg[i];
  consumer_bar();
  const uint32_t lpp = hd / 4, ppw = 32 / lpp;
  const uint32_t sub = lane % lpp, slot = lane / lpp, e0 = sub * 4;
  const int64_t q0 = q_s[e0], q1 = q_s[e0 + 1], q2 = q_s[e0 + 2], q3 = q_s[e0 + 3];
  // stage 0: scores ((q . k) >> 16) * inv >> 24 and their maximum
  long long lmax = LLONG_MIN;
  for (uint32_t base = warp * ppw; base < nsc; base += kNCW * ppw) {
    const uint32_t tl = base + slot;
    unsigned long long d = 0;
    if (tl < nsc) {
      const int4 k4 = *reinterpret_cast<const int4*>(Kh + (size_t)(s0 + tl) * p.kv_dim + e0);
      d = (unsigned long long)q0 * (unsigned long long)(long long)k4.x +
          (unsigned long long)q1 * (unsigned long long)(long long)k4.y +
          (unsigned long long)q2 * (unsigned long long)(long long)k4.z +
          (unsigned long long)q3 * (unsigned long long)(long long)k4.w;
    }
    for (uint32_t o = lpp >> 1; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (tl < nsc && sub == 0) {
      long long s = (long long)d >> 16;
      s = (long long)((unsigned long long)s * (unsigned long long)p.inv_sqrt) >> 24;
      sc[tl] = s;
      lmax = s > lmax ? s : lmax;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const long long t = __shfl_xor_sync(0xffffffffu, lmax, o);
    lmax = t > lmax ? t : lmax;
  }
  if (lane == 0) red[warp] = lmax;
  consumer_bar();
  long long m = LLONG_MIN;
  for (int w = 0; w < kNCW; ++w) m = red[w] > m ? red[w] : m;
  if (!full) {
    if (tid == 0) parts[2 * ch] = m;
    if (!group_sync(q, sh, hcount, (2 * l + 1) * gh)) return false;
    m = LLONG_MIN;
    for (uint32_t j = 0; j < gh; ++j) {
      const long long v = *(volatile long long*)(parts + 2 * j);
      m = v > m ? v : m;
    }
  }
  // stage 1: exponentials EXP[min((m - s) >> 8, 4096)] and their sum
  unsigned long long z = 0;
  for (uint32_t tl = tid; tl < nsc; tl += kCT) {
    unsigned long long idx = ((unsigned long long)m - (unsigned long long)sc[tl]) >> 8;
    if (idx > 4096) idx = 4096;
    const unsigned long long e = __ldg(p.exp_tab + idx);
    sc[tl] = (long long)e;
    z += e;
  }
  z = warp_sum(z);
  consumer_bar();  // every warp has read red (the maximum) before it is reused
  if (lane == 0) red[warp] = (long long)z;
  consumer_bar();
  unsigned long long Z = 0;
  for (int w = 0; w < kNCW; ++w) Z += (unsigned long long)red[w];
  if (!full) {
    if (tid == 0) parts[2 * ch + 1] = (long long)Z;
    if (!group_sync(q, sh, hcount, (2 * l + 2) * gh)) return false;
    Z = 0;
    for (uint32_t j = 0; j < gh; ++j) Z += (unsigned long long)*(volatile long long*)(parts + 2 * j + 1);
  }
  // stage 2: probabilities (e << 24) / Z over this CTA's chunk [t0, t1)
  const bool small_z = Z > 0 && Z <= 0xFFFFFFFFull;
  const InvDiv DZ = make_invdiv(small_z ? (uint32_t)Z : 1u);
  for (uint32_t t = t0 + tid; t < t1; t += kCT) {
    const unsigned long long num = (unsigned long long)sc[t - s0] << 24;
    sc[t - s0] = (long long)(small_z ? udiv_inv(num, DZ) : num / Z);
  }
  consumer_bar();
  // stage 3: sum over the chunk of P * v, added into the head's accumulators
  const uint32_t nch = t1 - t0;
  unsigned long long a0 = 0, a1 = 0, a2 = 0, a3 = 0;
  for (uint32_t base = warp * ppw; base < nch; base += kNCW * ppw) {
    const uint32_t tl = base + slot;
    if (tl < nch) {
      const int4 v4 = *reinterpret_cast<const int4*>(Vh + (size_t)(t0 + tl) * p.kv_dim + e0);
      const long long pr = sc[t0 - s0 + tl];
      a0 += (unsigned long long)(pr * (long long)v4.x);
      a1 += (unsigned long long)(pr * (long long)v4.y);
      a2 += (unsigned long long)(pr * (long long)v4.z);
      a3 += (unsigned long long)(pr * (long long)v4.w);
    }
  }
  for (uint32_t o = 16; o >= lpp && o > 0; o >>= 1) {
    a0 += __shfl_xor_sync(0xffffffffu, a0, o);
    a1 += __shfl_xor_sync(0xffffffffu, a1, o);
    a2 += __shfl_xor_sync(0xffffffffu, a2, o);
    a3 += __shfl_xor_sync(0xffffffffu, a3, o);
  }
  if (slot == 0) {
    unsigned long long* dst = part + (size_t)warp * hd + e0;
    dst[0] = a0;
    dst[1] = a1;
    dst[2] = a2;
    dst[3] = a3;
  }
  consumer_bar();
  if (nch) {
    unsigned long long* acc = reinterpret_cast<unsigned long long*>(q.work + p.off_oacc) + (size_t)h * hd;
    for (uint32_t j = tid; j < hd; j += kCT) {
      unsigned long long s = 0;
      for (int w = 0; w < kNCW; ++w) s += part[(size_t)w * hd + j];
      if (gh == 1) acc[j] = s;  // the only contributor
      else atomicAdd(acc + j, s);
    }
  }
  return true;
}

// ------------------------------------------------------------------ the position


__device__ __forceinline__ void consumers(const StepParams& p, const Pos& q, Shared& sh) {
  uint32_t epoch = 0;
  RingPos rp = {0u, 0u};
  Best best;
  best.v = LLONG_MIN;
  best.i = 0xFFFFFFFFu;
  for (uint32_t l = 0; l <= p.layers; ++l) {
    for (int k = kQKV; k <= kDOWN; ++k) {
      int kind = k;
      if (l == p.layers) {
        if (k > kQKV) break;
        kind = p.generating ? kCLS : kEND;
      }
      if (!(l == 0 && kind == kQKV) && !grid_sync(q, sh, epoch)) return;
      if (kind == kEND) return;
      if (kind == kATT) {
        if (!attention(p, q, l, sh)) return;
        continue;
      }
      const MR m = matrow_of(p, q, l < p.layers ? l : 0, kind);
      unsigned long long S;
      uint32_t lcap;
      const int L = prologue(p, q, m, sh, &S, &lcap);
      consume_phase(p, q, m, l, L, S, lcap, rp, sh, best);
      consumer_bar();
      if (sh.abort) return;
      if (kind == kCLS) {
        // this CTA's first largest logit, then the grid's in the last phase
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          Best ob;
          ob.v = __shfl_xor_sync(0xffffffffu, best.v, o);
          ob.i = __shfl_xor_sync(0xffffffffu, best.i, o);
          if (ob.i != 0xFFFFFFFFu) best_update(best, ob.v, ob.i);
        }
        if (lane == 0) {
          sh.am_v[warp] = best.v;
          sh.am_i[warp] = best.i;
        }
        consumer_bar();
        long long* cand = reinterpret_cast<long long*>(q.work + p.off_cand);
        if (threadIdx.x == 0) {
          Best cb;
          cb.v = LLONG_MIN;
          cb.i = 0xFFFFFFFFu;
          for (int w = 0; w < kNCW; ++w)
            if (sh.am_i[w] != 0xFFFFFFFFu) best_update(cb, sh.am_v[w], sh.am_i[w]);
          cand[2 * blockIdx.x] = cb.v;
          cand[2 * blockIdx.x + 1] = (long long)cb.i;
        }
        if (!grid_sync(q, sh, epoch)) return;
        if (blockIdx.x != 0) return;
        // phase 19 (maximum pass over the per-CTA candidates) and the end of the position
        if (threadIdx.x == 0) {
          Best g;
          g.v = LLONG_MIN;
          g.i = 0xFFFFFFFFu;
          for (uint32_t b = 0; b < gridDim.x; ++b) {
            const long long v = *(volatile const long long*)(cand + 2 * b);
            const uint32_t i = (uint32_t) * (volatile const long long*)(cand + 2 * b + 1);
            if (i != 0xFFFFFFFFu) best_update(g, v, i);
          }
          uint8_t* st = p.st;
          if (hdr_ld<uint64_t>(st, kHErrKey) != kNoError) {
            hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
            hdr<uint32_t>(st, kHError) = CK_ARITHMETIC;
          } else {
            const uint32_t gen = hdr_ld<uint32_t>(st, kHGenerated);
            reinterpret_cast<uint32_t*>(st + p.off_out)[gen] = g.i;
            hdr<uint32_t>(st, kHGenerated) = gen + 1;
            hdr<uint32_t>(st, kHLastTok) = g.i;
            hdr<long long>(st, kHMaxLogit) = g.v;
            const bool stop =
                (hdr_ld<uint32_t>(st, kHFlags) & CK_FLAG_STOP_TOKENS) && (g.i == 1 || g.i == 2);
            if (gen + 1 == hdr_ld<uint32_t>(st, kHMaxTok) || stop) hdr<uint32_t>(st, kHPhase) = CK_PHASE_DONE;
            hdr<uint32_t>(st, kHPosition) += 1;
          }
        }
        return;
      }
    }
  }
}

// The whole position for one CTA, with its scratch at `work`.
__device__ __forceinline__ void step_body(const StepParams& p, uint8_t* work, Shared& sh) {
  uint8_t* st = p.st;
  if (hdr_ld<uint32_t>(st, kHPhase) != CK_PHASE_RUNNING) return;  // every CTA alike
  Pos q;
  q.work = work;
  q.pos = hdr_ld<uint32_t>(st, kHPosition);
  const uint32_t np = hdr_ld<uint32_t>(st, kHNPrompt);
  q.tok = q.pos < np ? reinterpret_cast<const uint32_t*>(st + p.off_prompt)[q.pos]
                     : reinterpret_cast<const uint32_t*>(st + p.off_out)[q.pos - np];
  if (q.tok >= p.vocab) {  // a state edited outside the library
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      hdr<uint32_t>(st, kHError) = CK_INVALID_STATE;
      hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
    }
    return;
  }
  if (threadIdx.x == 0) {
    sh.abort = 0;
    for (uint32_t s = 0; s < p.ns; ++s) {
      mbar_init(&full_of(p)[s], 1);
      mbar_init(&empty_of(p)[s], kNCW);  // every consumer warp releases every slot
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if ((threadIdx.x >> 5) == kNCW) {
    if ((threadIdx.x & 31) == 0) producer(p, q);
    return;
  }
  consumers(p, q, sh);
  // a prompt position ends with the last residual and the cursor (block 0, after the grid
  // barrier the consumers passed on their way out of the last layer)
  if (!p.generating && blockIdx.x == 0 && !sh.abort) {
    int64_t* x = reinterpret_cast<int64_t*>(st + p.off_x);
    const int64_t* xb = reinterpret_cast<const int64_t*>(st + p.off_xb);
    const int64_t* y = reinterpret_cast<const int64_t*>(st + p.off_y);
    for (uint32_t i = threadIdx.x; i < p.dim; i += kCT) x[i] = wadd(xb[i], y[i]);
    if (threadIdx.x == 0) {
      if (hdr_ld<uint64_t>(st, kHErrKey) != kNoError) {
        hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
        hdr<uint32_t>(st, kHError) = CK_ARITHMETIC;
      } else {
        hdr<uint32_t>(st, kHPosition) += 1;
      }
    }
  }
  if (threadIdx.x == 0 && blockIdx.x == 0 && (sh.abort || ld_acquire(gabort_of(q)))) {
    hdr<uint32_t>(st, kHError) = CK_CUDA_ERROR;
    hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
  }
}

__global__ void __launch_bounds__(kThreads, 1) k_step(const StepParams p) {
  __shared__ Shared sh;
  step_body(p, p.st + p.off_work, sh);
}

// ------------------------------------------------------------------ allocation-free variant
// The same position with its scratch (barrier counters, attention partials and
// accumulators, classifier candidates, global planes) in this file's own device array
// instead of the state's work region.
constexpr size_t kNoAllocWorkBytes = 256 * 1024;
static __device__ __align__(256) uint8_t g_noalloc_work[kNoAllocWorkBytes];

__global__ void __launch_bounds__(kThreads, 1) k_step_noalloc(const StepParams p, uint8_t* work) {
  __shared__ Shared sh;
  step_body(p, work, sh);
}

cudaError_t launch_coop(const void* fn, void** args, cudaStream_t s, int grid, size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

size_t noalloc_work_bytes() { return kNoAllocWorkBytes; }

// Set-up of the allocation-free variant, once per device, with that device current: the
// device address of the scratch array (host code only holds a stand-in for the symbol) and
// the kernel's shared-memory limit.  Later calls on the device reuse the cached address.
cudaError_t noalloc_setup(size_t dynamic_max, uint8_t** work) {
  static uint8_t* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_work);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_step_noalloc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dynamic_max);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<uint8_t*>(ptr);
  }
  *work = addr[dev];
  return cudaSuccess;
}

cudaError_t launch_step_noalloc(const StepParams& p, uint8_t* work, cudaStream_t s, int grid, size_t smem) {
  StepParams pc = p;
  uint8_t* w = work;
  void* args[2] = {&pc, &w};
  return launch_coop(reinterpret_cast<const void*>(k_step_noalloc), args, s, grid, smem);
}

// Allows the kernel the largest dynamic shared memory the device offers beside its static
// shared memory; *dynamic_max receives that size.
cudaError_t configure_step(size_t optin, size_t* dynamic_max) {
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, k_step);
  if (e != cudaSuccess) return e;
  if (optin <= a.sharedSizeBytes) return cudaErrorInvalidValue;
  *dynamic_max = optin - a.sharedSizeBytes;
  return cudaFuncSetAttribute(k_step, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)*dynamic_max);
}

cudaError_t launch_step(const StepParams& p, cudaStream_t s, int grid, size_t smem) {
  StepParams pc = p;
  void* args[1] = {&pc};
  return launch_coop(reinterpret_cast<const void*>(k_step), args, s, grid, smem);
}

int step_threads() { return kThreads; }

int step_blocks_per_sm(size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_step, kThreads, smem) != cudaSuccess) return 0;
  return n;
}
int step_consumer_warps() { return kNCW; }
size_t step_red_bytes() { return (size_t)kNCW * kPanelRows * 8; }

}  // namespace ck
