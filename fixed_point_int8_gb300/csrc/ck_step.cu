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
#include <mutex>

#include "ck_internal.cuh"

namespace ck {
namespace {

constexpr int kNCW = (int)kStepWarps;   // consumer warps
constexpr int kCT = 32 * kNCW;          // consumer threads
constexpr int kThreads = kCT + 32;      // plus one producer warp
constexpr uint32_t kPollLimit = 1u << 22;
constexpr int kRMax = (int)(kPanelRows / 32);  // rows a lane accumulates

// work area offsets (bytes from the start of the state's scores/work region); the first
// zero_bytes are cleared before every launch
constexpr uint32_t kWBar = 0, kWAbort = 4;  // then the per-vector sums (8 .. 80)

enum Epi : int { kEResid = 0, kEQKV = 1, kESiLU = 2, kELogits = 3 };
enum Kind : int { kQKV = 0, kATT = 1, kO = 2, kGU = 3, kDOWN = 4, kCLS = 5, kEND = 6 };

struct MR {
  const uint8_t* W;  // column-group layout
  const uint32_t* scale;
  uint32_t pitch, rows, cols;
  uint32_t vin;               // index of the input vector (see "phase inputs")
  int epi;
  int64_t* out;               // Q/K/V: the rotated queries; classifier: the logits
  int32_t* kc;                // Q/K/V: this layer's key and value cache
  int32_t* vc;
  const int64_t* res_in;      // O, DOWN: the residual stream the outputs add to
  int64_t* res_out;           // O, DOWN: the sum (the next norm's input)
  const int32_t* next_norm;   // O, DOWN: the next norm's weights (nullptr: none)
};

struct Shared {
  unsigned long long ra[kNCW], rbuf[kNCW];
  long long am_v[kNCW];
  uint32_t am_i[kNCW];
  unsigned long long smp_state, smp_sum, smp_draw;  // phase 19 above temperature zero
  unsigned long long S, orv;
  int abort;
  int last;
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
  uint32_t sync_polls;  // polls of a grid or head-group barrier before it gives up
};
__device__ __forceinline__ uint32_t* gbar_of(const Pos& q) { return reinterpret_cast<uint32_t*>(q.work + kWBar); }
__device__ __forceinline__ uint32_t* gabort_of(const Pos& q) { return reinterpret_cast<uint32_t*>(q.work + kWAbort); }

__device__ __forceinline__ int64_t* st64(const StepParams& p, uint64_t off) {
  return reinterpret_cast<int64_t*>(p.st + off);
}

// The matrix-row phase of kind `k` in layer l ("The forward pass, in order"):
//   QKV   the attention norm's output times Wq, Wk, Wv; rotary on Q and K, checked cache
//         stores of K and V
//   O     the head outputs times Wo; x + y goes to xb (the feed-forward norm's input)
//   GU    the feed-forward norm's output times the gate and up rows; SiLU gating gives h
//   DOWN  h times W2; xb + y goes to x (the next layer's, or the final, norm's input)
//   CLS   the final norm's output times the classifier rows into the logits
__device__ __forceinline__ MR matrow_of(const StepParams& p, const Pos& q, uint32_t l, int k) {
  MR m = {};
  const DevLayer* W = p.layers_tab + l;
  int64_t* x = st64(p, p.off_x);
  int64_t* xb = st64(p, p.off_xb);
  if (k == kQKV) {
    m.W = W->wqkv; m.scale = W->sqkv; m.pitch = p.pitch_d; m.rows = p.dim + 2 * p.kv_dim; m.cols = p.dim;
    m.vin = 4 * l; m.epi = kEQKV; m.out = st64(p, p.off_q);
    const size_t lw = (size_t)p.cache * p.kv_dim;
    m.kc = reinterpret_cast<int32_t*>(p.st + p.off_k) + l * lw;
    m.vc = reinterpret_cast<int32_t*>(p.st + p.off_v) + l * lw;
  } else if (k == kO) {
    m.W = W->wo; m.scale = W->so; m.pitch = p.pitch_d; m.rows = p.dim; m.cols = p.dim;
    m.vin = 4 * l + 1; m.epi = kEResid; m.res_in = x; m.res_out = xb; m.next_norm = W->ffn_norm;
  } else if (k == kGU) {
    m.W = W->w13; m.scale = W->s13; m.pitch = p.pitch_d; m.rows = 2 * p.hidden; m.cols = p.dim;
    m.vin = 4 * l + 2; m.epi = kESiLU;
  } else if (k == kDOWN) {
    m.W = W->w2; m.scale = W->s2; m.pitch = p.pitch_h; m.rows = p.dim; m.cols = p.hidden;
    m.vin = 4 * l + 3; m.epi = kEResid; m.res_in = xb; m.res_out = x;
    m.next_norm = l + 1 < p.layers ? W[1].attn_norm : (p.generating ? p.final_norm : nullptr);
  } else {  // classifier
    m.W = p.cls; m.scale = p.cls_scale; m.pitch = p.pitch_d; m.rows = p.vocab; m.cols = p.dim;
    m.vin = 4 * p.layers; m.epi = kELogits; m.out = st64(p, p.off_logits);
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

// The producer warp: fills ring slot gs % ns with stage gs once the slot's previous stage
// is released (lane 0 waits and arms the slot's barrier, then lane j issues the bulk copy
// of the stage's group j), and optionally keeps L2 prefetches of the following stages
// about pf_bytes ahead of the fills, so that HBM keeps streaming while the consumers are in
// barriers, prologues or attention and the ring is full.
__device__ void producer(const StepParams& p, const Pos& q) {
  const uint32_t lane = threadIdx.x & 31;
  uint64_t* full = full_of(p);
  const uint32_t ns = p.ns;
  StageCursor fc, pc;
  cursor_start(p, q, fc);
  cursor_start(p, q, pc);
  unsigned long long filled = 0, fetched = 0;  // bytes
  uint32_t gs = 0, slot = 0, epar = 0;  // epar: parity of the slot's previous release
  bool stop = false;
  for (; !fc.done; cursor_next(p, q, fc), ++gs) {
    const uint32_t run = fc.pn * kGroupCols;
    const uint32_t ng = min(fc.gps, fc.NG - fc.g0);
    const size_t gstride = (size_t)fc.rows * kGroupCols;
    // prefetch ahead (the fill cursor never passes the prefetch cursor)
    while (p.pf_bytes && !pc.done && fetched < filled + ng * run + p.pf_bytes) {
      const uint32_t prun = pc.pn * kGroupCols, png = min(pc.gps, pc.NG - pc.g0);
      const uint8_t* src = pc.W + (size_t)(pc.rb + pc.p0) * kGroupCols + (size_t)pc.g0 * pc.rows * kGroupCols;
      for (uint32_t gl = lane; gl < png; gl += 32) prefetch_l2(src + (size_t)gl * pc.rows * kGroupCols, prun);
      fetched += (unsigned long long)png * prun;
      cursor_next(p, q, pc);
    }
    if (lane == 0) {
      if (gs >= ns) {
        if (!producer_wait_empty(p, q, slot, epar)) {
          stop = true;
        } else if (!mbar_try(&full[slot], epar)) {
          atomicExch(gabort_of(q), 1u);  // the slot's last fill never completed: stop, do not re-arm
          stop = true;
        }
      }
      if (!stop) mbar_expect_tx(&full[slot], ng * run);
    }
    stop = __shfl_sync(0xffffffffu, stop ? 1 : 0, 0) != 0;
    if (stop) break;
    for (uint32_t gl = lane; gl < ng; gl += 32) {  // small panels put many groups in a stage
      uint8_t* dst = ring_of() + (size_t)slot * kStageBytes + (size_t)gl * run;
      const uint8_t* src = fc.W + (size_t)(fc.rb + fc.p0) * kGroupCols + (size_t)(fc.g0 + gl) * gstride;
      bulk_g2s(dst, src, run, &full[slot]);
    }
    filled += (unsigned long long)ng * run;
    if (++slot == ns) {  // stage gs + 1 = k ns: from k = 2 on, each wrap flips the parity
      slot = 0;
      if (gs + 1 > ns) epar ^= 1u;
    }
  }
  // wait (bounded) for every copy still in flight before the CTA may exit
  if (lane == 0) {
    for (uint32_t j = gs > ns ? gs - ns : 0; j < gs; ++j) {
      for (uint32_t i = 0; i < kPollLimit; ++i)
        if (mbar_try(&full[j % ns], (j / ns) & 1)) break;
    }
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
      if (++i > q.sync_polls || ((i & 255) == 0 && ld_acquire(gabort_of(q)))) {
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
      if (++i > q.sync_polls || ((i & 255) == 0 && ld_acquire(gabort_of(q)))) {
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

// ------------------------------------------------------------------ phase inputs
// Every matrix phase reads its input vector (index vin: 4l + 0 the attention norm's output,
// 4l + 1 the head outputs, 4l + 2 the feed-forward norm's output, 4l + 3 h, 4L the final
// norm's output) as byte planes: plane k holds byte k of every element.  The planes sit in
// one of three global buffers (vin mod 3), written by the blocks that produce the elements,
// together with two sums over the vector (the wrapping sum S for the -128 * S correction
// and the OR of |x| that sets the limb count); a phase starts with one bulk copy of them
// into shared memory.  Norm inputs also need the wrapping sum of squares SS of the
// residual they normalise, added up by the blocks that produce the residual.  The sums live
// in the cleared part of the work region in three slots (vin mod 3); the slot of vin + 2 is
// cleared while phase vin runs (its last readers finished before that phase's barrier, and
// its first writers come after the next one).
constexpr int kSumS = 0, kSumOr = 1, kSumSq = 2;
__device__ __forceinline__ unsigned long long* vsum(const Pos& q, int kind, uint32_t vin) {
  return reinterpret_cast<unsigned long long*>(q.work + 8) + 3 * kind + vin % 3;
}
__device__ __forceinline__ unsigned long long vsum_ld(const Pos& q, int kind, uint32_t vin) {
  return *reinterpret_cast<volatile unsigned long long*>(vsum(q, kind, vin));
}
__device__ __forceinline__ uint8_t* vbuf(const StepParams& p, const Pos& q, uint32_t vin) {
  return q.work + p.off_vbuf + (size_t)(vin % 3) * 8 * p.vbuf_pitch;
}
__device__ __forceinline__ uint64_t* pbar_of(const StepParams& p) { return empty_of(p) + p.ns; }

// The eight bytes of v into planes 0..7 at column c.
__device__ __forceinline__ void put_planes(uint8_t* buf, uint32_t pitch, uint32_t c, int64_t v) {
#pragma unroll
  for (int k = 0; k < 8; ++k) buf[(size_t)k * pitch + c] = (uint8_t)((uint64_t)v >> (8 * k));
}

// Limb count of a vector from the OR of |x|: 1 to 4, or 8 (the consumers' bodies).
__device__ __forceinline__ int limbs_of(unsigned long long orv) {
  int L = 1;
  while (L < 8 && (orv >> (8 * L - 1)) != 0) ++L;
  return L > 4 ? 8 : L;
}

// Adds this block's partial sums of a vector into its slot (one atomic each).
__device__ void add_vector_sums(const Pos& q, uint32_t vin, unsigned long long s, unsigned long long o,
                                Shared& sh) {
  consumer_sum_or(s, o, sh);
  if (threadIdx.x == 0) {
    atomicAdd(vsum(q, kSumS, vin), s);
    atomicOr(vsum(q, kSumOr, vin), o);
  }
}

__device__ __forceinline__ void mbar_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
               : "memory");
}

// "RMS normalization" of this block's slice of a norm input: rms = isqrt(SS/n + 42,950),
// at least 1, then y = ((x * w) / rms) >> 8 with the division truncating toward zero, from
// the residual slice and the weights staged in shared memory; the bytes of y go to the
// vector's planes and the block's sums to its slot.
__device__ void distribute(const StepParams& p, const Pos& q, uint32_t vin, Shared& sh) {
  uint32_t rb, re;
  cta_rows(p.dim, blockIdx.x, gridDim.x, rb, re);
  const int64_t* vs = reinterpret_cast<const int64_t*>(xreg(p) + p.x_vslice);
  const int32_t* ws = reinterpret_cast<const int32_t*>(xreg(p) + p.x_wslice);
  uint64_t rms = isqrt_u64(udiv_inv(vsum_ld(q, kSumSq, vin), p.div_dim) + 42950ull);
  if (rms < 1) rms = 1;
  const InvDiv D = make_invdiv((uint32_t)rms);
  uint8_t* buf = vbuf(p, q, vin);
  unsigned long long S = 0, orv = 0;
  for (uint32_t t = threadIdx.x; t < re - rb; t += kCT) {
    const int64_t y = sdiv_trunc(wmul(vs[t], (int64_t)ws[t]), D) >> 8;
    put_planes(buf, p.pitch_d, rb + t, y);
    S += (unsigned long long)y;
    orv |= (unsigned long long)(y ^ (y >> 63));
  }
  add_vector_sums(q, vin, S, orv, sh);
}

// Vector 0, phase 3 and the first attention norm: every block adds up the squares of the
// whole embedding row itself (it is only dim bytes), then writes its slice of the residual
// x = ((byte - 128) * scale) >> 8 and of the normalised planes.
__device__ void distribute_embed(const StepParams& p, const Pos& q, Shared& sh) {
  const int64_t s = (int64_t)__ldg(p.embed_scale + q.tok);
  unsigned long long ss = 0, dummy = 0;
  for (uint32_t e0 = 16 * threadIdx.x; e0 < p.dim; e0 += 16 * kCT) {
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(p.embed + grouped_offset(p.vocab, q.tok, e0)));
    const uint32_t wd[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int64_t x = ((int64_t)((wd[i >> 2] >> (8 * (i & 3))) & 0xFFu) - 128) * s >> 8;
      if (e0 + i < p.dim) ss += (unsigned long long)x * (unsigned long long)x;
    }
  }
  consumer_sum_or(ss, dummy, sh);
  uint64_t rms = isqrt_u64(udiv_inv(ss, p.div_dim) + 42950ull);
  if (rms < 1) rms = 1;
  const InvDiv D = make_invdiv((uint32_t)rms);
  uint32_t rb, re;
  cta_rows(p.dim, blockIdx.x, gridDim.x, rb, re);
  int64_t* x = st64(p, p.off_x);
  const int32_t* w = p.layers_tab[0].attn_norm;
  uint8_t* buf = vbuf(p, q, 0);
  unsigned long long S = 0, orv = 0;
  for (uint32_t r = rb + threadIdx.x; r < re; r += kCT) {
    const int64_t xv = ((int64_t)p.embed[grouped_offset(p.vocab, q.tok, r)] - 128) * s >> 8;
    x[r] = xv;
    const int64_t y = sdiv_trunc(wmul(xv, (int64_t)__ldg(w + r)), D) >> 8;
    put_planes(buf, p.pitch_d, r, y);
    S += (unsigned long long)y;
    orv |= (unsigned long long)(y ^ (y >> 63));
  }
  add_vector_sums(q, 0, S, orv, sh);
}

// Start of a matrix phase: one bulk copy of the input's planes 0..3 into shared memory
// (and 4..7 when the vector needs more than four limbs and they fit), the vector's sums,
// this block's row scales and (Q/K/V) the position's rotary row, and (O, DOWN) the residual
// slice the outputs add to with the next norm's weights for it.  Block 0 also clears the
// sums' slot of vector vin + 2 and, for Q/K/V, the attention accumulators.  Returns the
// limb count; *S_out the wrapping sum, *lcap_out the planes held in shared memory.
__device__ int fetch_prologue(const StepParams& p, const Pos& q, const MR& m, Shared& sh, uint32_t& ppar,
                              unsigned long long* S_out, uint32_t* lcap_out) {
  const uint32_t pitch = m.pitch, tid = threadIdx.x;
  uint32_t lcap = p.planes_bytes / pitch;
  if (lcap > 8) lcap = 8;
  uint32_t rb, re;
  cta_rows(m.rows, blockIdx.x, gridDim.x, rb, re);
  uint8_t* X = xreg(p);
  uint32_t* sc = reinterpret_cast<uint32_t*>(X + p.planes_bytes);
  int32_t* rp = reinterpret_cast<int32_t*>(X + p.planes_bytes + 4 * p.scale_cap);
  int64_t* vs = reinterpret_cast<int64_t*>(X + p.x_vslice);
  int32_t* ws = reinterpret_cast<int32_t*>(X + p.x_wslice);
  const bool qkv = m.epi == kEQKV;
  uint64_t* pbar = pbar_of(p);
  const uint8_t* src = vbuf(p, q, m.vin);
  if (tid == 0) {
    // the planes were written by other blocks' generic stores before the grid barrier
    asm volatile("fence.proxy.async.global;" ::: "memory");
    mbar_expect(pbar, 4 * pitch);
    bulk_g2s(X, src, 4 * pitch, pbar);
  }
  // loads whose results are only stored at the end: in flight during the rest
  const uint32_t my_row = rb + tid;
  const uint32_t my_scale = my_row < re ? __ldg(m.scale + my_row) : 0u;
  const int32_t my_rope = (qkv && tid < p.hd) ? __ldg(p.rope + (size_t)q.pos * p.hd + tid) : 0;
  const unsigned long long S = vsum_ld(q, kSumS, m.vin);
  const int L = limbs_of(vsum_ld(q, kSumOr, m.vin));
  if (tid == 0) {
    if (L > 4 && lcap > 4) {
      const uint32_t nb = (lcap - 4) * pitch;
      mbar_expect(pbar, nb);
      bulk_g2s(X + 4 * pitch, src + 4 * pitch, nb, pbar);
    }
    mbar_arrive(pbar);
  }
  if (blockIdx.x == 0) {
    if (tid < 3) *vsum(q, (int)tid, m.vin + 2) = 0ull;
    if (qkv) {
      unsigned long long* acc = reinterpret_cast<unsigned long long*>(q.work + p.off_oacc);
      for (uint32_t i = tid; i < p.dim; i += kCT) acc[i] = 0ull;
    }
  }
  if (m.epi == kEResid) {
    for (uint32_t t = tid; t < re - rb; t += kCT) {
      vs[t] = m.res_in[rb + t];
      ws[t] = m.next_norm ? __ldg(m.next_norm + rb + t) : 0;
    }
  }
  if (my_row < re) sc[tid] = my_scale;
  for (uint32_t r = my_row + kCT; r < re; r += kCT) sc[r - rb] = __ldg(m.scale + r);
  if (qkv && tid < p.hd) rp[tid] = my_rope;
  for (uint32_t i = tid + kCT; qkv && i < p.hd; i += kCT) rp[i] = __ldg(p.rope + (size_t)q.pos * p.hd + i);
  bool ok = false;
  for (uint32_t i = 0; i < kPollLimit; ++i) {
    if (mbar_try(pbar, ppar)) {
      ok = true;
      break;
    }
  }
  ppar ^= 1u;
  if (!ok) {
    atomicExch(gabort_of(q), 1u);
    sh.abort = 1;
  }
  consumer_bar();  // the scales, rotary row and slices of the other threads
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

// Per-thread partial sums of the vector an epilogue produces (see "phase inputs").
struct OutSums {
  unsigned long long s, o, sq;
};

// Epilogue of one row (threads with valid == false only take part in the partner exchange;
// the partner of an even row is the next thread).  t is the row's index in this CTA's
// slice.
__device__ __forceinline__ void epilogue(const StepParams& p, const Pos& q, const MR& m, uint32_t layer,
                                         uint32_t row, uint32_t t, bool valid, int64_t y, Best& best,
                                         const int32_t* rope, int64_t* vs, OutSums& os) {
  const int64_t partner = (int64_t)__shfl_xor_sync(0xffffffffu, (unsigned long long)y, 1);
  if (!valid) return;
  if (m.epi == kEResid) {
    // the residual: its sum goes on, to be normalised by the next phase
    const int64_t v = wadd(vs[t], y);
    m.res_out[row] = v;
    vs[t] = v;
    os.sq += (unsigned long long)v * (unsigned long long)v;
  } else if (m.epi == kELogits) {
    m.out[row] = y;
    best_update(best, y, row);
  } else if (m.epi == kESiLU) {
    if ((row & 1) == 0) {
      // h = (silu(gate) * up) >> 16, straight into the planes of DOWN's input
      const int64_t h = wmul(silu_lookup(y, p.silu_tab), partner) >> 16;
      put_planes(vbuf(p, q, m.vin + 1), p.pitch_h, row >> 1, h);
      os.s += (unsigned long long)h;
      os.o |= (unsigned long long)(h ^ (h >> 63));
    }
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
      m.kc[cache_word(e, q.pos, p.hd, p.cache)] = (int32_t)mine;
    } else {
      const uint32_t e = row - q_rows - p.kv_dim;
      if (!fits_i32(y)) record_error(p.st, err_key(q.pos, layer, 7, e));
      m.vc[cache_word(e, q.pos, p.hd, p.cache)] = (int32_t)y;
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
  const uint8_t* gpl = vbuf(p, q, m.vin) + (size_t)lcap * pitch;  // planes lcap.. in global memory
  const uint32_t* sc = reinterpret_cast<const uint32_t*>(xreg(p) + p.planes_bytes);
  const int32_t* rope = reinterpret_cast<const int32_t*>(xreg(p) + p.planes_bytes + 4 * p.scale_cap);
  int64_t* vs = reinterpret_cast<int64_t*>(xreg(p) + p.x_vslice);
  unsigned long long* red = red_of(p);
  OutSums os = {0ull, 0ull, 0ull};
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
    epilogue(p, q, m, layer, rb + p0 + tid, p0 + tid, valid, y, best, rope, vs, os);
    consumer_bar();  // every thread has read the partial sums before the next panel's
  }
  // this block's share of the sums of the vector the phase produced
  if (m.epi == kESiLU) {
    add_vector_sums(q, m.vin + 1, os.s, os.o, sh);
  } else if (m.epi == kEResid && m.next_norm) {
    unsigned long long dummy = 0;
    consumer_sum_or(os.sq, dummy, sh);
    if (tid == 0) atomicAdd(vsum(q, kSumSq, m.vin + 1), os.sq);
  }
}

// ------------------------------------------------------------------ attention

constexpr int kAB = 8;  // positions a lane group loads at once: one memory round trip each

// Stage 0 over positions [s0, s0 + n): scores ((q . k) >> 16) * inv >> 24 into sc, lanes
// along the head dimension (hd / 4 lanes a position, four elements each), kAB positions a
// lane group per round so that all of a round's key loads are in flight together.
// Returns the thread's largest score (LLONG_MIN if none).
__device__ __forceinline__ long long att_scores(const StepParams& p, const int32_t* Kh, uint32_t s0, uint32_t n,
                                                const int64_t* q_s, long long* sc) {
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lpp = p.hd / 4, ppw = 32 / lpp, sub = lane % lpp, slot = lane / lpp, e0 = sub * 4;
  const int64_t q0 = q_s[e0], q1 = q_s[e0 + 1], q2 = q_s[e0 + 2], q3 = q_s[e0 + 3];
  long long lmax = LLONG_MIN;
  const uint32_t round = kNCW * ppw * kAB;
  for (uint32_t base = 0; base < n; base += round) {
    int4 k4[kAB];
#pragma unroll
    for (int bb = 0; bb < kAB; ++bb) {
      const uint32_t tl = base + (bb * kNCW + warp) * ppw + slot;
      k4[bb] = tl < n ? *reinterpret_cast<const int4*>(Kh + (size_t)(s0 + tl) * p.hd + e0) : make_int4(0, 0, 0, 0);
    }
    unsigned long long d[kAB];
#pragma unroll
    for (int bb = 0; bb < kAB; ++bb)
      d[bb] = (unsigned long long)q0 * (unsigned long long)(long long)k4[bb].x +
              (unsigned long long)q1 * (unsigned long long)(long long)k4[bb].y +
              (unsigned long long)q2 * (unsigned long long)(long long)k4[bb].z +
              (unsigned long long)q3 * (unsigned long long)(long long)k4[bb].w;
    for (uint32_t o = lpp >> 1; o > 0; o >>= 1) {
#pragma unroll
      for (int bb = 0; bb < kAB; ++bb) d[bb] += __shfl_xor_sync(0xffffffffu, d[bb], o);
    }
#pragma unroll
    for (int bb = 0; bb < kAB; ++bb) {
      const uint32_t tl = base + (bb * kNCW + warp) * ppw + slot;
      if (tl < n && sub == 0) {
        long long sv = (long long)d[bb] >> 16;
        sv = (long long)((unsigned long long)sv * (unsigned long long)p.inv_sqrt) >> 24;
        sc[tl] = sv;
        lmax = sv > lmax ? sv : lmax;
      }
    }
  }
  return lmax;
}

// Stage 3 over positions [t0, t0 + n) and dimensions [dlo, dlo + dn) (dn a multiple of 4):
// the wrapping sums over positions of P_t * v_t, lanes along the dimensions, kAB positions
// a lane group per round; the warp's sums over its positions end in part[warp][0 .. dn).
__device__ __forceinline__ void att_values(const StepParams& p, const int32_t* Vh, uint32_t t0, uint32_t n,
                                           uint32_t dlo, uint32_t dn, const long long* pr,
                                           unsigned long long* part) {
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lpp = dn / 4, ppw = 32 / lpp, sub = lane % lpp, slot = lane / lpp, e0 = sub * 4;
  unsigned long long a0 = 0, a1 = 0, a2 = 0, a3 = 0;
  const uint32_t round = kNCW * ppw * kAB;
  for (uint32_t base = 0; base < n; base += round) {
    int4 v4[kAB];
    long long pb[kAB];
#pragma unroll
    for (int bb = 0; bb < kAB; ++bb) {
      const uint32_t tl = base + (bb * kNCW + warp) * ppw + slot;
      v4[bb] = tl < n ? *reinterpret_cast<const int4*>(Vh + (size_t)(t0 + tl) * p.hd + dlo + e0)
                      : make_int4(0, 0, 0, 0);
      pb[bb] = tl < n ? pr[tl] : 0;
    }
#pragma unroll
    for (int bb = 0; bb < kAB; ++bb) {
      a0 += (unsigned long long)(pb[bb] * (long long)v4[bb].x);
      a1 += (unsigned long long)(pb[bb] * (long long)v4[bb].y);
      a2 += (unsigned long long)(pb[bb] * (long long)v4[bb].z);
      a3 += (unsigned long long)(pb[bb] * (long long)v4[bb].w);
    }
  }
  for (uint32_t o = 16; o >= lpp && o > 0; o >>= 1) {
    a0 += __shfl_xor_sync(0xffffffffu, a0, o);
    a1 += __shfl_xor_sync(0xffffffffu, a1, o);
    a2 += __shfl_xor_sync(0xffffffffu, a2, o);
    a3 += __shfl_xor_sync(0xffffffffu, a3, o);
  }
  if (slot == 0) {
    unsigned long long* dst = part + (size_t)warp * dn + e0;
    dst[0] = a0;
    dst[1] = a1;
    dst[2] = a2;
    dst[3] = a3;
  }
}

// O's input elements o = sum >> 24 of head dimensions [c0, c0 + cn): byte planes and this
// block's part of the vector's sums.
__device__ __forceinline__ void att_output(const StepParams& p, const Pos& q, uint32_t l, uint32_t c0, uint32_t cn,
                                           const unsigned long long* sums, Shared& sh) {
  uint8_t* buf = vbuf(p, q, 4 * l + 1);
  unsigned long long S = 0, orv = 0;
  for (uint32_t j = threadIdx.x; j < cn; j += kCT) {
    const int64_t o = (int64_t)sums[j] >> 24;
    put_planes(buf, p.pitch_d, c0 + j, o);
    S += (unsigned long long)o;
    orv |= (unsigned long long)(o ^ (o >> 63));
  }
  add_vector_sums(q, 4 * l + 1, S, orv, sh);
}

// Phase 9 for this CTA's (head, share): "Attention" in four stages over positions 0..pos
// of the head's cache.  The maximum and the sum Z need every position.  Short contexts
// (up to att_full positions): every CTA of the head scores all positions itself and takes
// a share of the head's dimensions in stage 3, so its outputs are final.  Longer ones: the
// CTAs score their own chunks of positions, exchange maxima and sums (two barriers among
// the head's CTAs), add sum_t P_t * v_t over their chunks into the head's 64-bit
// accumulators, and the last to finish turns them into the outputs.
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
  const uint32_t s0 = full ? 0u : t0, nsc = (full ? P : t1) - s0;
  const uint32_t kvh = h / (p.heads / p.kv_heads);
  const size_t lw = (size_t)p.cache * p.kv_dim;
  // the head's positions are one contiguous run of the head-major cache
  const int32_t* Kh = reinterpret_cast<const int32_t*>(p.st + p.off_k) + l * lw + (size_t)kvh * p.cache * hd;
  const int32_t* Vh = reinterpret_cast<const int32_t*>(p.st + p.off_v) + l * lw + (size_t)kvh * p.cache * hd;
  long long* parts = reinterpret_cast<long long*>(q.work + p.off_part) + (size_t)h * gh * 2;  // [gh][2]
  uint32_t* hcount = reinterpret_cast<uint32_t*>(q.work + p.off_hsync) + h;
  const int64_t* qg = st64(p, p.off_q) + (size_t)h * hd;
  for (uint32_t i = tid; i < hd; i += kCT) q_s[i] = qg[i];
  consumer_bar();
  // stage 0: scores and their maximum
  long long lmax = att_scores(p, Kh, s0, nsc, q_s, sc);
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
  // stage 2: probabilities (e << 24) / Z over the positions stage 3 needs
  const uint32_t v0 = full ? 0u : t0, nv = full ? P : t1 - t0;
  const bool small_z = Z > 0 && Z <= 0xFFFFFFFFull;
  const InvDiv DZ = make_invdiv(small_z ? (uint32_t)Z : 1u);
  for (uint32_t t = tid; t < nv; t += kCT) {
    const unsigned long long num = (unsigned long long)sc[v0 - s0 + t] << 24;
    sc[v0 - s0 + t] = (long long)(small_z ? udiv_inv(num, DZ) : num / Z);
  }
  consumer_bar();
  if (full) {
    // stage 3 on this CTA's share of the head's dimensions: final outputs
    const uint32_t nsplit = min(gh, hd / 4), dn = hd / nsplit;
    if (ch >= nsplit) return true;
    att_values(p, Vh, 0, P, ch * dn, dn, sc, part);
    consumer_bar();
    unsigned long long* fin = reinterpret_cast<unsigned long long*>(q_s);  // [dn]: q is no longer needed
    for (uint32_t j = tid; j < dn; j += kCT) {
      unsigned long long v = 0;
      for (int w = 0; w < kNCW; ++w) v += part[(size_t)w * dn + j];
      fin[j] = v;
    }
    consumer_bar();
    att_output(p, q, l, h * hd + ch * dn, dn, fin, sh);
    return true;
  }
  // stage 3 on this CTA's chunk of positions, added into the head's accumulators
  att_values(p, Vh, t0, t1 - t0, 0, hd, sc + (t0 - s0), part);
  consumer_bar();
  unsigned long long* acc = reinterpret_cast<unsigned long long*>(q.work + p.off_oacc) + (size_t)h * hd;
  if (t1 > t0) {
    for (uint32_t j = tid; j < hd; j += kCT) {
      unsigned long long v = 0;
      for (int w = 0; w < kNCW; ++w) v += part[(size_t)w * hd + j];
      atomicAdd(acc + j, v);
    }
  }
  // the head's last CTA to finish turns the accumulators into O's input
  __threadfence();
  consumer_bar();
  if (tid == 0) {
    uint32_t* fin = reinterpret_cast<uint32_t*>(q.work + p.off_hfin) + h;
    sh.last = atomicAdd(fin, 1u) == (l + 1) * gh - 1;
  }
  consumer_bar();
  if (sh.last) {
    __threadfence();
    unsigned long long* fin = part;  // [hd], reused
    for (uint32_t j = tid; j < hd; j += kCT) fin[j] = *reinterpret_cast<volatile unsigned long long*>(acc + j);
    consumer_bar();
    att_output(p, q, l, h * hd, hd, fin, sh);
  }
  return true;
}

// ------------------------------------------------------------------ the position


// One matrix phase: prologue (planes of its input), the rows, the epilogues.  False on abort.
__device__ __forceinline__ bool matrix_phase(const StepParams& p, const Pos& q, uint32_t l, int kind,
                                             RingPos& rp, uint32_t& ppar, Shared& sh, Best& best) {
  const MR m = matrow_of(p, q, l, kind);
  unsigned long long S;
  uint32_t lcap;
  const int L = fetch_prologue(p, q, m, sh, ppar, &S, &lcap);
  consume_phase(p, q, m, l, L, S, lcap, rp, sh, best);
  consumer_bar();
  return sh.abort == 0;
}

// The consumer warps' sequence for one position (grid barriers between dependent steps):
//   embedding and first attention norm (every block its slice)
//   per layer: QKV | attention (+ O's input) | O (+ residual) | norm slices | GU (+ h) |
//              DOWN (+ residual) | next norm slices
//   when the position generates: final norm slices | classifier | maximum pass
__device__ __forceinline__ void consumers(const StepParams& p, const Pos& q, Shared& sh) {
  uint32_t epoch = 0, ppar = 0;
  RingPos rp = {0u, 0u};
  Best best;
  best.v = LLONG_MIN;
  best.i = 0xFFFFFFFFu;
  distribute_embed(p, q, sh);
  if (!grid_sync(q, sh, epoch)) return;
  for (uint32_t l = 0; l < p.layers; ++l) {
    if (!matrix_phase(p, q, l, kQKV, rp, ppar, sh, best)) return;
    if (!grid_sync(q, sh, epoch)) return;
    if (!attention(p, q, l, sh)) return;
    if (!grid_sync(q, sh, epoch)) return;
    if (!matrix_phase(p, q, l, kO, rp, ppar, sh, best)) return;
    if (!grid_sync(q, sh, epoch)) return;
    distribute(p, q, 4 * l + 2, sh);
    if (!grid_sync(q, sh, epoch)) return;
    if (!matrix_phase(p, q, l, kGU, rp, ppar, sh, best)) return;
    if (!grid_sync(q, sh, epoch)) return;
    if (!matrix_phase(p, q, l, kDOWN, rp, ppar, sh, best)) return;
    if (!grid_sync(q, sh, epoch)) return;
    if (l + 1 < p.layers || p.generating) {
      distribute(p, q, 4 * l + 4, sh);
      if (!grid_sync(q, sh, epoch)) return;
    }
  }
  if (!p.generating) return;  // a prompt position: x holds the last residual
  if (!matrix_phase(p, q, 0, kCLS, rp, ppar, sh, best)) return;
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
  // phase 19: maximum pass over the per-CTA candidates
  if (threadIdx.x == 0) {
    Best g;
    g.v = LLONG_MIN;
    g.i = 0xFFFFFFFFu;
    for (uint32_t b = 0; b < gridDim.x; ++b) {
      const long long v = *(volatile const long long*)(cand + 2 * b);
      const uint32_t i = (uint32_t) * (volatile const long long*)(cand + 2 * b + 1);
      if (i != 0xFFFFFFFFu) best_update(g, v, i);
    }
    sh.am_v[0] = g.v;
    sh.am_i[0] = g.i;
    sh.smp_state = hdr_ld<unsigned long long>(p.st, kHSeed);
    sh.smp_sum = 0;
    sh.smp_draw = 0;
  }
  const uint32_t temp = hdr_ld<uint32_t>(p.st, kHTemp);
  if (temp == 0) return;
  // sum and draw passes by block 0's consumer warps; the ring's shared memory is free now
  consumer_bar();
  const SampleOut so = block_sample(reinterpret_cast<const long long*>(st64(p, p.off_logits)),
                                    p.vocab, sh.am_v[0], temp, p.exp_tab, sh.smp_state,
                                    reinterpret_cast<unsigned long long*>(ring_of()), kNCW,
                                    [] { consumer_bar(); });
  if (threadIdx.x == 0) {
    sh.am_i[0] = so.token;
    sh.smp_state = so.state;
    sh.smp_sum = so.sum;
    sh.smp_draw = so.draw;
  }
}

// The whole position for one CTA, with its scratch at `work`.
__device__ __forceinline__ void step_body(const StepParams& p, uint8_t* work, Shared& sh) {
  uint8_t* st = p.st;
  if (hdr_ld<uint32_t>(st, kHPhase) != CK_PHASE_RUNNING) return;  // every CTA alike
  Pos q;
  q.work = work;
  q.sync_polls = p.sync_polls ? p.sync_polls : kPollLimit;
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
    mbar_init(pbar_of(p), 1);  // the phase prologue's plane copy
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if ((threadIdx.x >> 5) == kNCW) {
    producer(p, q);
    return;
  }
  consumers(p, q, sh);
  // block 0 ends the position after the last grid barrier: the generated token (phase 19)
  // or, for a prompt position, only the cursor; a failed cache store fails the state
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  if (sh.abort || ld_acquire(gabort_of(q))) {
    hdr<uint32_t>(st, kHError) = CK_CUDA_ERROR;
    hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
    return;
  }
  if (hdr_ld<uint64_t>(st, kHErrKey) != kNoError) {
    hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
    hdr<uint32_t>(st, kHError) = CK_ARITHMETIC;
    return;
  }
  if (p.generating) {
    const uint32_t tok = sh.am_i[0];
    const uint32_t gen = hdr_ld<uint32_t>(st, kHGenerated);
    reinterpret_cast<uint32_t*>(st + p.off_out)[gen] = tok;
    hdr<uint32_t>(st, kHGenerated) = gen + 1;
    hdr<uint32_t>(st, kHLastTok) = tok;
    hdr<long long>(st, kHMaxLogit) = sh.am_v[0];
    hdr<unsigned long long>(st, kHSeed) = sh.smp_state;
    hdr<unsigned long long>(st, kHExpSum) = sh.smp_sum;
    hdr<unsigned long long>(st, kHDraw) = sh.smp_draw;
    const bool stop = (hdr_ld<uint32_t>(st, kHFlags) & CK_FLAG_STOP_TOKENS) && (tok == 1 || tok == 2);
    if (gen + 1 == hdr_ld<uint32_t>(st, kHMaxTok) || stop) hdr<uint32_t>(st, kHPhase) = CK_PHASE_DONE;
  }
  hdr<uint32_t>(st, kHPosition) += 1;
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
// A mutex makes the first call on a device run the set-up once even when several host
// threads make it at the same time.
cudaError_t noalloc_setup(size_t dynamic_max, uint8_t** work) {
  static std::mutex mu;
  static uint8_t* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
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
