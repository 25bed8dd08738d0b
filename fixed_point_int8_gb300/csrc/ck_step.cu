// One position of the forward pass ("The inference core", "The forward pass, in order") as
// one persistent kernel: one CTA per SM, launched cooperatively so every CTA is resident.
//
// GB300 design.  Each CTA owns a contiguous slice of the rows of every matrix of the step.
// A producer warp streams those slices, matrix after matrix and layer after layer, through
// a ring of shared-memory slots with cp.async.bulk copies completing on mbarriers; it never
// waits for activations, only for free slots, so HBM keeps streaming across phase
// boundaries.  Eight consumer warps own ring stages round-robin; for each matrix they pack
// the phase's input vector into byte planes (after the residual and the RMS
// normalization where the phase has them), run the dp4a matrix-row loop on the staged rows
// and apply the fused epilogue.  Phases that depend on each other are separated by a grid
// barrier among the consumer warps.  Attention splits each head's positions over a few
// CTAs that exchange their maxima, sums and partial weighted values through the state's
// work area behind per-head group barriers.  Every wait is bounded: on a timeout the kernel
// raises an abort flag, stops issuing copies, waits (bounded) for its copies in flight and
// the state is marked failed with error 9.
#include <climits>

#include "ck_internal.cuh"

namespace ck {
namespace {

constexpr int kNCW = 8;                 // consumer warps
constexpr int kCT = 32 * kNCW;          // consumer threads
constexpr int kThreads = kCT + 32;      // plus one producer warp
constexpr uint32_t kPollLimit = 1u << 22;

// work area offsets (bytes from the start of the state's scores/work region)
constexpr uint32_t kWBar = 0, kWAbort = 4, kWHeads = 64, kWPart = 4096;  // [0, 4096) zeroed per launch

enum Pro : int { kPPlain = 0, kPNorm = 1, kPEmbedNorm = 2 };
enum Epi : int { kEStore = 0, kEQKV = 1, kESiLU = 2, kELogits = 3 };
enum Kind : int { kQKV = 0, kATT = 1, kO = 2, kGU = 3, kDOWN = 4, kCLS = 5, kEND = 6 };

struct MR {
  const uint8_t* W;
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
  const uint32_t* scales;  // this block's row scales of the phase (shared memory)
  const int32_t* rope;     // this position's (cos, sin) pairs (shared memory)
  uint32_t rb;             // first row of this block in the phase
  unsigned long long ra[kNCW], rbuf[kNCW];
  long long am_v[kNCW];
  uint32_t am_i[kNCW];
  InvDiv div;
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

struct Ctx {
  const StepParams* p;
  uint8_t* st;
  uint8_t* work;
  uint32_t* gbar;
  uint32_t* gabort;
  uint8_t* ring;
  uint8_t* X;
  uint64_t* full;
  uint64_t* empty;
  uint32_t ns, pos, tok, G;
};

__device__ __forceinline__ int64_t* st64(const Ctx& c, uint64_t off) {
  return reinterpret_cast<int64_t*>(c.st + off);
}

// The matrix-row phase of kind `k` in layer l (see the phase table in the design notes).
__device__ MR matrow_of(const Ctx& c, uint32_t l, int k) {
  const StepParams& p = *c.p;
  MR m = {};
  const DevLayer* W = p.layers_tab + l;
  int64_t* x = st64(c, p.off_x);
  int64_t* xb = st64(c, p.off_xb);
  int64_t* y = st64(c, p.off_y);
  if (k == kQKV) {
    m.W = W->wqkv; m.scale = W->sqkv; m.pitch = p.pitch_d; m.rows = p.dim + 2 * p.kv_dim; m.cols = p.dim;
    m.pro = l == 0 ? kPEmbedNorm : kPNorm;
    m.in = xb; m.add = l == 0 ? nullptr : y; m.res_out = x; m.norm_w = W->attn_norm;
    m.epi = kEQKV; m.out = st64(c, p.off_q);
    const size_t lw = (size_t)p.cache * p.kv_dim;
    m.kc = reinterpret_cast<int32_t*>(c.st + p.off_k) + l * lw;
    m.vc = reinterpret_cast<int32_t*>(c.st + p.off_v) + l * lw;
  } else if (k == kO) {
    m.W = W->wo; m.scale = W->so; m.pitch = p.pitch_d; m.rows = p.dim; m.cols = p.dim;
    m.pro = kPPlain; m.in = st64(c, p.off_o); m.epi = kEStore; m.out = y;
  } else if (k == kGU) {
    m.W = W->w13; m.scale = W->s13; m.pitch = p.pitch_d; m.rows = 2 * p.hidden; m.cols = p.dim;
    m.pro = kPNorm; m.in = x; m.add = y; m.res_out = xb; m.norm_w = W->ffn_norm;
    m.epi = kESiLU; m.out = st64(c, p.off_h);
  } else if (k == kDOWN) {
    m.W = W->w2; m.scale = W->s2; m.pitch = p.pitch_h; m.rows = p.dim; m.cols = p.hidden;
    m.pro = kPPlain; m.in = st64(c, p.off_h); m.epi = kEStore; m.out = y;
  } else {  // classifier
    m.W = p.cls; m.scale = p.cls_scale; m.pitch = p.pitch_d; m.rows = p.vocab; m.cols = p.dim;
    m.pro = kPNorm; m.in = xb; m.add = y; m.res_out = x; m.norm_w = p.final_norm;
    m.epi = kELogits; m.out = st64(c, p.off_logits);
  }
  return m;
}

// This CTA's rows of a matrix: whole pairs, split evenly over the grid.
__device__ __forceinline__ void cta_rows(const MR& m, uint32_t b, uint32_t G, uint32_t& rb, uint32_t& re) {
  const uint32_t np = (m.rows + 1) / 2;
  const uint32_t pb = (uint32_t)((uint64_t)np * b / G), pe = (uint32_t)((uint64_t)np * (b + 1) / G);
  rb = min(m.rows, 2 * pb);
  re = min(m.rows, 2 * pe);
}
__device__ __forceinline__ uint32_t stage_rows(uint32_t pitch) {
  uint32_t sr = kStageBytes / pitch;
  if (sr >= 2) sr &= ~1u;
  return sr < 1 ? 1 : sr;
}

// ------------------------------------------------------------------ producer

__device__ bool producer_wait_empty(const Ctx& c, uint32_t slot, uint32_t parity) {
  for (uint32_t i = 0; i < kPollLimit; ++i) {
    if (mbar_try(&c.empty[slot], parity)) return true;
    if ((i & 63) == 63 && ld_acquire(c.gabort)) return false;
  }
  atomicExch(c.gabort, 1u);
  return false;
}

__device__ void producer(const Ctx& c) {
  const StepParams& p = *c.p;
  uint32_t gs = 0;
  bool ok = true;
  for (uint32_t l = 0; l <= p.layers && ok; ++l) {
    for (int kk = 0; kk < 4 && ok; ++kk) {
      int k = kk == 0 ? kQKV : kk == 1 ? kO : kk == 2 ? kGU : kDOWN;
      if (l == p.layers) {
        if (!p.generating || kk > 0) break;
        k = kCLS;
      }
      const MR m = matrow_of(c, l < p.layers ? l : 0, k);
      uint32_t rb, re;
      cta_rows(m, blockIdx.x, c.G, rb, re);
      const uint32_t sr = stage_rows(m.pitch);
      for (uint32_t r0 = rb; r0 < re; r0 += sr, ++gs) {
        const uint32_t slot = gs % c.ns;
        if (gs >= c.ns && !producer_wait_empty(c, slot, ((gs / c.ns) - 1) & 1)) {
          ok = false;
          break;
        }
        if (gs >= c.ns && !mbar_try(&c.full[slot], ((gs / c.ns) - 1) & 1)) {
          atomicExch(c.gabort, 1u);  // the slot's last fill never completed: stop, do not re-arm
          ok = false;
          break;
        }
        const uint32_t nr = min(sr, re - r0);
        mbar_expect_tx(&c.full[slot], nr * m.pitch);
        bulk_g2s(c.ring + (size_t)slot * kStageBytes, m.W + (size_t)r0 * m.pitch, nr * m.pitch,
                 &c.full[slot]);
      }
    }
  }
  // wait (bounded) for every copy still in flight before the CTA may exit
  for (uint32_t j = gs > c.ns ? gs - c.ns : 0; j < gs; ++j) {
    for (uint32_t i = 0; i < kPollLimit; ++i)
      if (mbar_try(&c.full[j % c.ns], (j / c.ns) & 1)) break;
  }
}

// ------------------------------------------------------------------ consumer helpers

// Barrier over the consumer warps of every CTA; `epoch` counts the barriers passed.
__device__ bool grid_sync(const Ctx& c, Shared& sh, uint32_t& epoch) {
  consumer_bar();
  ++epoch;
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(c.gbar) : "memory");
    const uint32_t target = epoch * c.G;
    uint32_t i = 0;
    while (ld_acquire(c.gbar) < target) {
      if (++i > kPollLimit || ld_acquire(c.gabort)) {
        atomicExch(c.gabort, 1u);
        sh.abort = 1;
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
  }
  consumer_bar();
  return sh.abort == 0;
}

// Barrier among the gh CTAs of one attention head (monotonic target within a launch).
__device__ bool group_sync(const Ctx& c, Shared& sh, uint32_t* counter, uint32_t target) {
  consumer_bar();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
    uint32_t i = 0;
    while (ld_acquire(counter) < target) {
      if (++i > kPollLimit || ld_acquire(c.gabort)) {
        atomicExch(c.gabort, 1u);
        sh.abort = 1;
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
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
  if (threadIdx.x == 0) {
    unsigned long long a = 0, b = 0;
    for (int w = 0; w < kNCW; ++w) {
      a += sh.ra[w];
      b |= sh.rbuf[w];
    }
    sh.S = a;
    sh.orv = b;
  }
  consumer_bar();
  s = sh.S;
  o = sh.orv;
}

constexpr int kPPT = 8;                                  // element pairs per thread per block
constexpr uint32_t kBlockPairs = (uint32_t)kCT * kPPT;   // 2048 pairs = 4096 elements

// The phase input for element pairs pbase + tid + j*kCT (j < kPPT): the embedding row of the
// token (phase 3), or in (+ add).  All loads of a block are issued before any is used, so a
// thread waits for one round trip per block instead of one per element.  Beyond n: zeros.
__device__ __forceinline__ void load_pairs(const Ctx& c, const MR& m, uint32_t pbase, int64_t (&x)[2 * kPPT]) {
  const uint32_t n = m.cols;
  if (m.pro == kPEmbedNorm) {
    const StepParams& p = *c.p;
    const uint8_t* row = p.embed + (size_t)c.tok * p.pitch_d;
    const int64_t s = (int64_t)__ldg(p.embed_scale + c.tok);
#pragma unroll
    for (int j = 0; j < kPPT; ++j) {
      const uint32_t i = 2 * (pbase + threadIdx.x + (uint32_t)j * kCT);
      int64_t a = 0, b = 0;
      if (i + 1 < n) {
        const uint16_t w = *reinterpret_cast<const uint16_t*>(row + i);
        a = ((int64_t)(w & 0xFF) - 128) * s >> 8;
        b = ((int64_t)(w >> 8) - 128) * s >> 8;
      } else if (i < n) {
        a = ((int64_t)row[i] - 128) * s >> 8;
      }
      x[2 * j] = a;
      x[2 * j + 1] = b;
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < kPPT; ++j) {
    const uint32_t i = 2 * (pbase + threadIdx.x + (uint32_t)j * kCT);
    int64_t a = 0, b = 0;
    if (i + 1 < n) {
      const longlong2 v = *reinterpret_cast<const longlong2*>(m.in + i);
      a = v.x;
      b = v.y;
    } else if (i < n) {
      a = m.in[i];
    }
    x[2 * j] = a;
    x[2 * j + 1] = b;
  }
  if (m.add) {
#pragma unroll
    for (int j = 0; j < kPPT; ++j) {
      const uint32_t i = 2 * (pbase + threadIdx.x + (uint32_t)j * kCT);
      if (i + 1 < n) {
        const longlong2 v = *reinterpret_cast<const longlong2*>(m.add + i);
        x[2 * j] = wadd(x[2 * j], v.x);
        x[2 * j + 1] = wadd(x[2 * j + 1], v.y);
      } else if (i < n) {
        x[2 * j] = wadd(x[2 * j], m.add[i]);
      }
    }
  }
}

// The norm weights of the same element pairs (zeros beyond n).
__device__ __forceinline__ void load_weights(const MR& m, uint32_t pbase, int2 (&w)[kPPT]) {
  const uint32_t n = m.cols;
#pragma unroll
  for (int j = 0; j < kPPT; ++j) {
    const uint32_t i = 2 * (pbase + threadIdx.x + (uint32_t)j * kCT);
    int2 v = make_int2(0, 0);
    if (i + 1 < n) v = *reinterpret_cast<const int2*>(m.norm_w + i);
    else if (i < n) v.x = m.norm_w[i];
    w[j] = v;
  }
}

// Packs the phase's input vector into byte planes (after the residual and the RMS
// normalization where the phase has them); returns the limb count and *S the wrapping sum.
__device__ int prologue(const Ctx& c, const MR& m, Shared& sh, unsigned long long* S_out) {
  const uint32_t n = m.cols, half = m.pitch / 2;
  const uint32_t npairs = (n + 1) / 2;
  uint16_t* planes16 = reinterpret_cast<uint16_t*>(c.X);
  const uint32_t lcap = c.p->lcap;
  uint16_t* gplanes16 = reinterpret_cast<uint16_t*>(c.work + c.p->off_gplanes);
  const bool writer = blockIdx.x == 0;
  const bool norm = m.pro != kPPlain;
  const bool single = half <= kBlockPairs;  // the whole vector fits one block of registers
  // this block's row scales (and for Q/K/V the position's rotary row) go to shared memory
  // so that no epilogue waits on global memory; the loads are issued first and stored last
  uint32_t rb, re;
  cta_rows(m, blockIdx.x, c.G, rb, re);
  uint32_t* sc = reinterpret_cast<uint32_t*>(c.X + c.p->planes_bytes);
  int32_t* rp = reinterpret_cast<int32_t*>(c.X + c.p->planes_bytes + 4 * c.p->scale_cap);
  const uint32_t my_row = rb + threadIdx.x;
  const uint32_t my_scale = my_row < re ? __ldg(m.scale + my_row) : 0u;
  const bool qkv = m.epi == kEQKV;
  const int32_t my_rope = (qkv && threadIdx.x < c.p->hd) ? __ldg(c.p->rope + (size_t)c.pos * c.p->hd + threadIdx.x) : 0;
  int64_t x[2 * kPPT];
  int2 wv[kPPT];
  if (norm) {
    // "RMS normalization": rms = isqrt(sum(x*x)/n + 42,950), at least 1
    unsigned long long ss = 0, dummy = 0;
    for (uint32_t pb = 0; pb < npairs; pb += kBlockPairs) {
      load_pairs(c, m, pb, x);
      if (single) load_weights(m, pb, wv);  // in flight while the sums reduce
#pragma unroll
      for (int e = 0; e < 2 * kPPT; ++e) ss += (unsigned long long)x[e] * (unsigned long long)x[e];
      if (writer && m.res_out) {
#pragma unroll
        for (int j = 0; j < kPPT; ++j) {
          const uint32_t i = 2 * (pb + threadIdx.x + (uint32_t)j * kCT);
          if (i + 1 < n) {
            longlong2 v;
            v.x = x[2 * j];
            v.y = x[2 * j + 1];
            *reinterpret_cast<longlong2*>(m.res_out + i) = v;
          } else if (i < n) {
            m.res_out[i] = x[2 * j];
          }
        }
      }
    }
    consumer_sum_or(ss, dummy, sh);
    if (threadIdx.x == 0) {
      const InvDiv& Dn = n == c.p->dim ? c.p->div_dim : c.p->div_hidden;
      uint64_t rms = isqrt_u64(udiv_inv(ss, Dn) + 42950ull);
      if (rms < 1) rms = 1;
      sh.div = make_invdiv((uint32_t)rms);
    }
    consumer_bar();
  }
  const InvDiv D = sh.div;
  unsigned long long S = 0, orv = 0;
  for (uint32_t pb = 0; pb < half; pb += kBlockPairs) {
    if (!(norm && single)) {  // a single block is still in registers
      load_pairs(c, m, pb, x);
      if (norm) load_weights(m, pb, wv);
    }
#pragma unroll
    for (int j = 0; j < kPPT; ++j) {
      const uint32_t pidx = pb + threadIdx.x + (uint32_t)j * kCT;
      if (pidx >= half) continue;
      const uint32_t i = 2 * pidx;
      int64_t v0 = x[2 * j], v1 = x[2 * j + 1];
      if (norm) {
        // y = ((x * w) / rms) >> 8, the division truncating toward zero
        v0 = i < n ? sdiv_trunc(wmul(v0, (int64_t)wv[j].x), D) >> 8 : 0;
        v1 = i + 1 < n ? sdiv_trunc(wmul(v1, (int64_t)wv[j].y), D) >> 8 : 0;
      }
      S += (unsigned long long)v0 + (unsigned long long)v1;
      orv |= (unsigned long long)(v0 ^ (v0 >> 63)) | (unsigned long long)(v1 ^ (v1 >> 63));
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if ((uint32_t)k >= lcap) break;
        planes16[(size_t)k * half + pidx] =
            (uint16_t)((((uint64_t)v0 >> (8 * k)) & 0xFF) | ((((uint64_t)v1 >> (8 * k)) & 0xFF) << 8));
      }
    }
  }
  if (my_row < re) sc[threadIdx.x] = my_scale;
  for (uint32_t r = my_row + kCT; r < re; r += kCT) sc[r - rb] = __ldg(m.scale + r);
  if (qkv && threadIdx.x < c.p->hd) rp[threadIdx.x] = my_rope;
  for (uint32_t i = threadIdx.x + kCT; qkv && i < c.p->hd; i += kCT)
    rp[i] = __ldg(c.p->rope + (size_t)c.pos * c.p->hd + i);
  if (threadIdx.x == 0) {
    sh.scales = sc;
    sh.rb = rb;
    sh.rope = rp;
  }
  consumer_sum_or(S, orv, sh);  // its barriers also publish the scales and the rotary row
  int L = 1;
  while (L < 8 && (orv >> (8 * L - 1)) != 0) ++L;
  if ((uint32_t)L > lcap) {
    // A vector beyond 8*lcap bits (rare): its planes lcap..L-1 go to the global copy, which
    // every block writes with the same bytes; the consumers read them from there.
    for (uint32_t pb = 0; pb < half; pb += kBlockPairs) {
      load_pairs(c, m, pb, x);
      if (norm) load_weights(m, pb, wv);
#pragma unroll
      for (int j = 0; j < kPPT; ++j) {
        const uint32_t pidx = pb + threadIdx.x + (uint32_t)j * kCT;
        if (pidx >= half) continue;
        const uint32_t i = 2 * pidx;
        int64_t v0 = x[2 * j], v1 = x[2 * j + 1];
        if (norm) {
          v0 = i < n ? sdiv_trunc(wmul(v0, (int64_t)wv[j].x), D) >> 8 : 0;
          v1 = i + 1 < n ? sdiv_trunc(wmul(v1, (int64_t)wv[j].y), D) >> 8 : 0;
        }
        for (uint32_t k = lcap; k < (uint32_t)L; ++k)
          gplanes16[(size_t)(k - lcap) * half + pidx] =
              (uint16_t)((((uint64_t)v0 >> (8 * k)) & 0xFF) | ((((uint64_t)v1 >> (8 * k)) & 0xFF) << 8));
      }
    }
    __threadfence_block();
    consumer_bar();
  }
  *S_out = S;
  return L;
}

// Row r (< 4) of the up to four rows a warp takes at once: the two rows of pair pq, then
// the two rows of pair pq + wg.
__device__ __forceinline__ uint32_t stage_row(uint32_t pq, uint32_t wg, uint32_t r) {
  return 2 * (pq + (r >> 1) * wg) + (r & 1);
}

// R rows of a stage (lanes along the row), rows stage_row(pq, wg, 0..R) of the stage;
// returns in lane r (< R) the 64-bit sum of row r.  Planes k < lcap are in shared memory, the others
// (only when kMixed) in the global copy.
template <int L, int R, bool kMixed>
__device__ __forceinline__ unsigned long long dot_rows(const uint8_t* stage, uint32_t pq, uint32_t wg,
                                                      uint32_t pitch, const uint8_t* planes_s,
                                                      const uint8_t* planes_g, uint32_t lcap) {
  const int lane = threadIdx.x & 31;
  const uint8_t* rp[R];
#pragma unroll
  for (int r = 0; r < R; ++r) rp[r] = stage + (size_t)stage_row(pq, wg, (uint32_t)r) * pitch;
  const uint8_t* pp[L];
#pragma unroll
  for (int k = 0; k < L; ++k)
    pp[k] = (!kMixed || (uint32_t)k < lcap) ? planes_s + (size_t)k * pitch : planes_g + (size_t)(k - lcap) * pitch;
  uint32_t acc[R][L];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int k = 0; k < L; ++k) acc[r][k] = 0;
  // Nine warps put three on one of the SM's four register-file quarters, which leaves 168
  // registers a thread: the column loop stays rolled so the accumulators never spill.
#pragma unroll 1
  for (uint32_t cc = lane * 16; cc < pitch; cc += 512) {
    uint4 w[R];
#pragma unroll
    for (int r = 0; r < R; ++r) w[r] = *reinterpret_cast<const uint4*>(rp[r] + cc);
#pragma unroll
    for (int k = 0; k < L; ++k) {
      const uint4 x = *reinterpret_cast<const uint4*>(pp[k] + cc);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (k < L - 1) {
          uint32_t a = acc[r][k];
          a = __dp4a(w[r].x, x.x, a);
          a = __dp4a(w[r].y, x.y, a);
          a = __dp4a(w[r].z, x.z, a);
          a = __dp4a(w[r].w, x.w, a);
          acc[r][k] = a;
        } else {
          int a = (int)acc[r][k];
          a = dp4a_us(w[r].x, x.x, a);
          a = dp4a_us(w[r].y, x.y, a);
          a = dp4a_us(w[r].z, x.z, a);
          a = dp4a_us(w[r].w, x.w, a);
          acc[r][k] = (uint32_t)a;
        }
      }
    }
  }
  unsigned long long mine = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    unsigned long long a = 0;
#pragma unroll
    for (int k = 0; k < L; ++k) {
      const unsigned long long t = (k < L - 1) ? (unsigned long long)acc[r][k]
                                               : (unsigned long long)(long long)(int)acc[r][k];
      a += t << (8 * k);
    }
    a = warp_sum(a);
    if (lane == r) mine = a;
  }
  return mine;
}

template <int L, bool kMixed>
__device__ __forceinline__ unsigned long long dot_rows_n(uint32_t R, const uint8_t* stage, uint32_t pq, uint32_t wg,
                                                        uint32_t pitch, const uint8_t* ps, const uint8_t* pg,
                                                        uint32_t lcap) {
  switch (R) {
    case 4: return dot_rows<L, 4, kMixed>(stage, pq, wg, pitch, ps, pg, lcap);
    case 3: return dot_rows<L, 3, kMixed>(stage, pq, wg, pitch, ps, pg, lcap);
    case 2: return dot_rows<L, 2, kMixed>(stage, pq, wg, pitch, ps, pg, lcap);
    default: return dot_rows<L, 1, kMixed>(stage, pq, wg, pitch, ps, pg, lcap);
  }
}

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

// Epilogue for the row of this lane (lanes < R), after the partner exchange for pairs.
__device__ __forceinline__ void epilogue(const Ctx& c, const MR& m, uint32_t layer, uint32_t row,
                                         bool valid, int64_t y, Best& best, const int32_t* rope) {
  const int64_t partner = (int64_t)__shfl_xor_sync(0xffffffffu, (unsigned long long)y, 1);
  if (!valid) return;
  const StepParams& p = *c.p;
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
      if (!fits_i32(y)) record_error(c.st, err_key(c.pos, layer, 6, e));
      const uint32_t j = (e % p.hd) >> 1;
      int64_t a2, b2;
      rotate_pair((int64_t)(int32_t)a, (int64_t)(int32_t)b, rope[2 * j], rope[2 * j + 1], a2, b2);
      const int64_t mine = even ? a2 : b2;
      if (!fits_i32(mine)) record_error(c.st, err_key(c.pos, layer, 8, e));
      m.kc[(size_t)c.pos * p.kv_dim + e] = (int32_t)mine;
    } else {
      const uint32_t e = row - q_rows - p.kv_dim;
      if (!fits_i32(y)) record_error(c.st, err_key(c.pos, layer, 7, e));
      m.vc[(size_t)c.pos * p.kv_dim + e] = (int32_t)y;
    }
  }
}

template <int L, bool kMixed>
__device__ void consume_phase(const Ctx& c, const MR& m, uint32_t layer, unsigned long long S,
                              uint32_t gs0, Shared& sh, Best& best) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const StepParams& p = *c.p;
  // Stages rotate over the warp groups; the warps of a group split each stage's row pairs.
  // A group's previous stage precedes the slot's previous use (groups <= slots), so its
  // parity wait can never see a phase two uses old.
  const uint32_t grp = (uint32_t)warp / p.wgroup, wi = (uint32_t)warp % p.wgroup;
  if (grp >= p.ngroups) return;
  uint32_t rb, re;
  cta_rows(m, blockIdx.x, c.G, rb, re);
  const uint32_t sr = stage_rows(m.pitch);
  const uint8_t* pg = c.work + p.off_gplanes;
  uint32_t gs = gs0;
  for (uint32_t r0 = rb; r0 < re; r0 += sr, ++gs) {
    if (gs % p.ngroups != grp) continue;
    const uint32_t slot = gs % c.ns;
    bool ok = false;
    for (uint32_t i = 0; i < kPollLimit; ++i) {
      if (mbar_try(&c.full[slot], (gs / c.ns) & 1)) {
        ok = true;
        break;
      }
      if ((i & 63) == 63 && ld_acquire(c.gabort)) break;
    }
    if (!ok) {
      atomicExch(c.gabort, 1u);
      sh.abort = 1;
      return;
    }
    const uint32_t nr = min(sr, re - r0);
    const uint32_t npairs = (nr + 1) / 2;
    const uint8_t* stage = c.ring + (size_t)slot * kStageBytes;
    // this warp's pairs: wi, wi + wgroup, ... taken two at a time (up to four rows)
    const uint32_t wg = p.wgroup;
    for (uint32_t pq = wi; pq < npairs; pq += 2 * wg) {
      // rows of pair pq, then of pair pq + wg; only the last pair of a stage can be single
      const uint32_t R = min(2 * pq + 2, nr) - 2 * pq + (pq + wg < npairs ? min(2 * (pq + wg) + 2, nr) - 2 * (pq + wg) : 0);
      const unsigned long long acc = dot_rows_n<L, kMixed>(R, stage, pq, wg, m.pitch, c.X, pg, p.lcap);
      const uint32_t row = r0 + stage_row(pq, wg, lane < 4 ? (uint32_t)lane : 0u);
      const bool valid = (uint32_t)lane < R;
      int64_t y = 0;
      if (valid) {
        const unsigned long long t = (acc - (S << 7)) * (unsigned long long)sh.scales[row - sh.rb];
        y = (int64_t)t >> 24;
      }
      epilogue(c, m, layer, row, valid, y, best, sh.rope);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.empty[slot]);
  }
}

__device__ uint32_t phase_stages(const Ctx& c, const MR& m) {
  uint32_t rb, re;
  cta_rows(m, blockIdx.x, c.G, rb, re);
  const uint32_t sr = stage_rows(m.pitch);
  return re > rb ? (re - rb + sr - 1) / sr : 0;
}

// Phase 9 for this CTA's (head, chunk).
__device__ bool attention(const Ctx& c, uint32_t l, Shared& sh) {
  const StepParams& p = *c.p;
  const uint32_t b = blockIdx.x, gh = p.gh;
  if (b >= p.heads * gh) return true;
  const uint32_t h = b / gh, ch = b % gh, hd = p.hd;
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int64_t* q_s = reinterpret_cast<int64_t*>(c.X);
  unsigned long long* part = reinterpret_cast<unsigned long long*>(q_s + hd);  // [kNCW][hd]
  long long* red = reinterpret_cast<long long*>(part + kNCW * hd);             // [kNCW]
  long long* sc = red + kNCW;                                                  // chunk scores
  const uint32_t P = c.pos + 1;
  const uint32_t cs = (P + gh - 1) / gh;
  const uint32_t t0 = min(P, ch * cs), t1 = min(P, t0 + cs), n = t1 - t0;
  const uint32_t kvh = h / (p.heads / p.kv_heads);
  const size_t lw = (size_t)p.cache * p.kv_dim;
  const int32_t* Kh = reinterpret_cast<const int32_t*>(c.st + p.off_k) + l * lw + (size_t)kvh * hd;
  const int32_t* Vh = reinterpret_cast<const int32_t*>(c.st + p.off_v) + l * lw + (size_t)kvh * hd;
  long long* wpart = reinterpret_cast<long long*>(c.work + kWPart) + (size_t)(h * gh + ch) * (hd + 2);
  uint32_t* hcount = reinterpret_cast<uint32_t*>(c.work + kWHeads) + h;
  const int64_t* qg = st64(c, p.off_q) + (size_t)h * hd;
  for (uint32_t i = tid; i < hd; i += kCT) q_s[i] = qg[i];
  consumer_bar();
  const uint32_t lpp = hd / 4, ppw = 32 / lpp;
  const uint32_t sub = lane % lpp, slot = lane / lpp, e0 = sub * 4;
  const int64_t q0 = q_s[e0], q1 = q_s[e0 + 1], q2 = q_s[e0 + 2], q3 = q_s[e0 + 3];
  // stage 0: scores ((q . k) >> 16) * inv >> 24 and the chunk maximum
  long long lmax = LLONG_MIN;
  for (uint32_t base = warp * ppw; base < n; base += kNCW * ppw) {
    const uint32_t tl = base + slot;
    unsigned long long d = 0;
    if (tl < n) {
      const int4 k4 = *reinterpret_cast<const int4*>(Kh + (size_t)(t0 + tl) * p.kv_dim + e0);
      d = (unsigned long long)q0 * (unsigned long long)(long long)k4.x +
          (unsigned long long)q1 * (unsigned long long)(long long)k4.y +
          (unsigned long long)q2 * (unsigned long long)(long long)k4.z +
          (unsigned long long)q3 * (unsigned long long)(long long)k4.w;
    }
    for (uint32_t o = lpp >> 1; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (tl < n && sub == 0) {
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
  if (gh > 1) {
    if (tid == 0) wpart[0] = m;
    if (!group_sync(c, sh, hcount, (3 * l + 1) * gh)) return false;
    m = LLONG_MIN;
    for (uint32_t j = 0; j < gh; ++j) {
      const long long v = *(volatile long long*)(reinterpret_cast<long long*>(c.work + kWPart) +
                                                 (size_t)(h * gh + j) * (hd + 2));
      m = v > m ? v : m;
    }
  }
  // stage 1: exponentials EXP[min((m - s) >> 8, 4096)] and their sum
  unsigned long long z = 0;
  for (uint32_t tl = tid; tl < n; tl += kCT) {
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
  if (gh > 1) {
    if (tid == 0) wpart[1] = (long long)Z;
    if (!group_sync(c, sh, hcount, (3 * l + 2) * gh)) return false;
    Z = 0;
    for (uint32_t j = 0; j < gh; ++j)
      Z += (unsigned long long)*(volatile long long*)(reinterpret_cast<long long*>(c.work + kWPart) +
                                                      (size_t)(h * gh + j) * (hd + 2) + 1);
  }
  // stage 2: probabilities (e << 24) / Z
  for (uint32_t tl = tid; tl < n; tl += kCT) sc[tl] = (long long)(((unsigned long long)sc[tl] << 24) / Z);
  consumer_bar();
  // stage 3: sum over positions of P * v, then one >> 24
  unsigned long long a0 = 0, a1 = 0, a2 = 0, a3 = 0;
  for (uint32_t base = warp * ppw; base < n; base += kNCW * ppw) {
    const uint32_t tl = base + slot;
    if (tl < n) {
      const int4 v4 = *reinterpret_cast<const int4*>(Vh + (size_t)(t0 + tl) * p.kv_dim + e0);
      const long long pr = sc[tl];
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
  int64_t* og = st64(c, p.off_o) + (size_t)h * hd;
  if (gh == 1) {
    for (uint32_t j = tid; j < hd; j += kCT) {
      unsigned long long s = 0;
      for (int w = 0; w < kNCW; ++w) s += part[(size_t)w * hd + j];
      og[j] = (int64_t)s >> 24;
    }
    return true;
  }
  for (uint32_t j = tid; j < hd; j += kCT) {
    unsigned long long s = 0;
    for (int w = 0; w < kNCW; ++w) s += part[(size_t)w * hd + j];
    wpart[2 + j] = (long long)s;
  }
  if (!group_sync(c, sh, hcount, (3 * l + 3) * gh)) return false;
  if (ch == 0) {
    for (uint32_t j = tid; j < hd; j += kCT) {
      unsigned long long s = 0;
      for (uint32_t q = 0; q < gh; ++q)
        s += (unsigned long long)*(volatile long long*)(reinterpret_cast<long long*>(c.work + kWPart) +
                                                        (size_t)(h * gh + q) * (hd + 2) + 2 + j);
      og[j] = (int64_t)s >> 24;
    }
  }
  return true;
}

__device__ void consumers(const Ctx& c, Shared& sh) {
  const StepParams& p = *c.p;
  uint32_t epoch = 0, gs = 0;
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
      if (!(l == 0 && kind == kQKV) && !grid_sync(c, sh, epoch)) return;
      if (kind == kEND) return;
      if (kind == kATT) {
        if (!attention(c, l, sh)) return;
        continue;
      }
      const MR m = matrow_of(c, l < p.layers ? l : 0, kind);
      unsigned long long S;
      const int L = prologue(c, m, sh, &S);
      const bool mixed = (uint32_t)L > p.lcap;
      switch (L) {
        case 1: consume_phase<1, false>(c, m, l, S, gs, sh, best); break;
        case 2: consume_phase<2, false>(c, m, l, S, gs, sh, best); break;
        case 3: consume_phase<3, false>(c, m, l, S, gs, sh, best); break;
        case 4: consume_phase<4, false>(c, m, l, S, gs, sh, best); break;
        case 5: mixed ? consume_phase<5, true>(c, m, l, S, gs, sh, best) : consume_phase<5, false>(c, m, l, S, gs, sh, best); break;
        case 6: mixed ? consume_phase<6, true>(c, m, l, S, gs, sh, best) : consume_phase<6, false>(c, m, l, S, gs, sh, best); break;
        case 7: mixed ? consume_phase<7, true>(c, m, l, S, gs, sh, best) : consume_phase<7, false>(c, m, l, S, gs, sh, best); break;
        default: mixed ? consume_phase<8, true>(c, m, l, S, gs, sh, best) : consume_phase<8, false>(c, m, l, S, gs, sh, best); break;
      }
      gs += phase_stages(c, m);
      consumer_bar();  // a warp that gave up returns early: leave together
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
        if (threadIdx.x == 0) {
          Best cb;
          cb.v = LLONG_MIN;
          cb.i = 0xFFFFFFFFu;
          for (int w = 0; w < kNCW; ++w)
            if (sh.am_i[w] != 0xFFFFFFFFu) best_update(cb, sh.am_v[w], sh.am_i[w]);
          long long* slot = reinterpret_cast<long long*>(c.work + kWPart) +
                            (size_t)p.heads * p.gh * (p.hd + 2) + 2 * blockIdx.x;
          slot[0] = cb.v;
          slot[1] = (long long)cb.i;
        }
        if (!grid_sync(c, sh, epoch)) return;
        if (blockIdx.x != 0) return;
        // phase 19 (maximum pass over the per-CTA candidates) and the end of the position
        if (threadIdx.x == 0) {
          Best g;
          g.v = LLONG_MIN;
          g.i = 0xFFFFFFFFu;
          const long long* slots = reinterpret_cast<const long long*>(c.work + kWPart) +
                                   (size_t)p.heads * p.gh * (p.hd + 2);
          for (uint32_t q = 0; q < c.G; ++q) {
            const long long v = *(volatile const long long*)(slots + 2 * q);
            const uint32_t i = (uint32_t) * (volatile const long long*)(slots + 2 * q + 1);
            if (i != 0xFFFFFFFFu) best_update(g, v, i);
          }
          uint8_t* st = c.st;
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

__global__ void __launch_bounds__(kThreads, 1) k_step(const StepParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ Shared sh;
  uint8_t* st = p.st;
  if (hdr_ld<uint32_t>(st, kHPhase) != CK_PHASE_RUNNING) return;  // every CTA alike
  Ctx c;
  c.p = &p;
  c.st = st;
  c.work = st + p.off_work;
  c.gbar = reinterpret_cast<uint32_t*>(c.work + kWBar);
  c.gabort = reinterpret_cast<uint32_t*>(c.work + kWAbort);
  c.ns = p.ns;
  c.G = gridDim.x;
  c.ring = smem;
  c.X = smem + (size_t)p.ns * kStageBytes;
  c.full = reinterpret_cast<uint64_t*>(c.X + p.x_bytes);
  c.empty = c.full + p.ns;
  c.pos = hdr_ld<uint32_t>(st, kHPosition);
  const uint32_t np = hdr_ld<uint32_t>(st, kHNPrompt);
  c.tok = c.pos < np ? reinterpret_cast<const uint32_t*>(st + p.off_prompt)[c.pos]
                     : reinterpret_cast<const uint32_t*>(st + p.off_out)[c.pos - np];
  if (c.tok >= p.vocab) {  // a state edited outside the library
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      hdr<uint32_t>(st, kHError) = CK_INVALID_STATE;
      hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
    }
    return;
  }
  if (threadIdx.x == 0) {
    sh.abort = 0;
    for (uint32_t s = 0; s < p.ns; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], p.wgroup);  // every warp of the owning group releases the slot
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if ((threadIdx.x >> 5) == kNCW) {
    if ((threadIdx.x & 31) == 0) producer(c);
    return;
  }
  consumers(c, sh);
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
  if (threadIdx.x == 0 && blockIdx.x == 0 && (sh.abort || ld_acquire(c.gabort))) {
    hdr<uint32_t>(st, kHError) = CK_CUDA_ERROR;
    hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
  }
}

// ------------------------------------------------------------------ allocation-free variant
// The same position with its scratch (barrier counters, attention partials, classifier
// candidates) in this file's own device array instead of the state's work region.
constexpr size_t kNoAllocWorkBytes = 256 * 1024;
static __device__ __align__(256) uint8_t g_noalloc_work[kNoAllocWorkBytes];

__global__ void __launch_bounds__(kThreads, 1) k_step_noalloc(const StepParams p, uint8_t* work) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ Shared sh;
  uint8_t* st = p.st;
  if (hdr_ld<uint32_t>(st, kHPhase) != CK_PHASE_RUNNING) return;
  Ctx c;
  c.p = &p;
  c.st = st;
  c.work = work;
  c.gbar = reinterpret_cast<uint32_t*>(c.work + kWBar);
  c.gabort = reinterpret_cast<uint32_t*>(c.work + kWAbort);
  c.ns = p.ns;
  c.G = gridDim.x;
  c.ring = smem;
  c.X = smem + (size_t)p.ns * kStageBytes;
  c.full = reinterpret_cast<uint64_t*>(c.X + p.x_bytes);
  c.empty = c.full + p.ns;
  c.pos = hdr_ld<uint32_t>(st, kHPosition);
  const uint32_t np = hdr_ld<uint32_t>(st, kHNPrompt);
  c.tok = c.pos < np ? reinterpret_cast<const uint32_t*>(st + p.off_prompt)[c.pos]
                     : reinterpret_cast<const uint32_t*>(st + p.off_out)[c.pos - np];
  if (c.tok >= p.vocab) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      hdr<uint32_t>(st, kHError) = CK_INVALID_STATE;
      hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
    }
    return;
  }
  if (threadIdx.x == 0) {
    sh.abort = 0;
    for (uint32_t s = 0; s < p.ns; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], p.wgroup);  // every warp of the owning group releases the slot
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if ((threadIdx.x >> 5) == kNCW) {
    if ((threadIdx.x & 31) == 0) producer(c);
    return;
  }
  consumers(c, sh);
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
  if (threadIdx.x == 0 && blockIdx.x == 0 && (sh.abort || ld_acquire(c.gabort))) {
    hdr<uint32_t>(st, kHError) = CK_CUDA_ERROR;
    hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
  }
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
  return cudaLaunchKernelEx(&cfg, k_step_noalloc, p, work);
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
  return cudaLaunchKernelEx(&cfg, k_step, p);
}

int step_threads() { return kThreads; }

int step_blocks_per_sm(size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_step, kThreads, smem) != cudaSuccess) return 0;
  return n;
}
int step_consumer_warps() { return kNCW; }

}  // namespace ck
