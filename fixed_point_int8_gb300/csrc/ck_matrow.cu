// The matrix-row kernel: y[r] = ((sum_c byte[r][c] * x[c] - 128 * sum_c x[c]) * scale[r]) >> 24
// with every product and sum wrapping in 64 bits ("The inference core", "A matrix row").
//
// GB300 design.  One CTA per SM (at most) takes an even-aligned share of the rows, so every
// SM streams even for 4,096-row matrices and both rows of a gate/up or rotary pair finish in
// the same CTA.  Its warps stream work items of 8 rows by a 512-byte column slice with 16-byte
// non-allocating loads, loading the next item while they work on the current one; the first
// item is requested before the vector is packed.  Before the rows, every CTA packs the input
// vector into shared memory as byte planes:
// plane k holds byte k of every x[c].  A vector whose values all fit in 8L signed bits is
// exactly sum_{k<L-1} plane_k 2^(8k) + signed(plane_{L-1}) 2^(8(L-1)), so
//   sum_c byte[r][c] * x[c] = sum_k 2^(8k) sum_c byte[r][c] * plane_k[c]
// where each inner sum is a run of dp4a (four u8 x u8 products per instruction, the top
// plane u8 x s8) into 32-bit accumulators that cannot overflow for cols <= 16384.  The
// limb count L is taken per vector from the OR of |x| (typically 3 for normalised inputs),
// so the ALU work is L/4 dp4a per weight byte instead of a 64-bit multiply-add per byte.
// The 64-bit result is then exact modulo 2^64, identical to the wrapping definition.
#include "ck_internal.cuh"

namespace ck {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kG = 8;                 // rows of one work item
constexpr uint32_t kSlice = 512;      // bytes of a row in one work item, 16 a lane
constexpr uint32_t kChunkRows = 256;  // rows a CTA finishes at once

struct Scratch {
  unsigned long long red[kWarps];
  unsigned long long red2[kWarps];
  InvDiv div;
  InvDiv divn;  // the vector length's reciprocal (norm prologue)
  unsigned long long S;
  unsigned long long orv;
  unsigned long long tot[kChunkRows];  // row totals of the current chunk
  long long res[kChunkRows];           // residual inputs of the chunk's rows (store epilogue)
};

// Programmatic dependent launch.  wait_prior_grids returns once the kernels before this one
// on the stream have completed and their writes are visible (at once when the launch did not
// allow an early start); allow_next_grid lets the next such kernel start its own independent
// prologue on SMs this grid frees.
__device__ __forceinline__ void wait_prior_grids() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 16- and 8-byte asynchronous copies from global to shared memory, and the wait for all of
// this thread's copies.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(src) : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

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

// Block-wide sum and OR (every thread gets both results).
__device__ void block_sum_or(unsigned long long& s, unsigned long long& o, Scratch* sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  s = warp_sum(s);
  o = warp_or(o);
  if (lane == 0) {
    sc->red[warp] = s;
    sc->red2[warp] = o;
  }
  __syncthreads();
  if (warp == 0) {
    unsigned long long a = lane < kWarps ? sc->red[lane] : 0ull;
    unsigned long long b = lane < kWarps ? sc->red2[lane] : 0ull;
    a = warp_sum(a);
    b = warp_or(b);
    if (lane == 0) {
      sc->S = a;
      sc->orv = b;
    }
  }
  __syncthreads();
  s = sc->S;
  o = sc->orv;
  __syncthreads();
}

__device__ __forceinline__ int64_t load_x(const MatrowParams& p, uint32_t i) {
  int64_t x = p.in[i];
  if (p.add) x = wadd(x, p.add[i]);
  return x;
}

// The prologue packs 4-element word groups: thread t takes groups t, t + kThreads, ...  Up to
// kPG groups a thread (8 elements: vectors of up to 4,096 elements at 512 threads) stay in
// registers from the sum of squares to the packing, and their norm weights are loaded before
// the kernel waits for the previous one (they are model data).
constexpr int kPG = 2;
constexpr int kPGP = 3;  // plain prologue: groups a thread loads at once (measured best of 2, 3, 6)

struct NormWeights {
  int32_t w[kPG][4];
};

// out[k] gets byte k of in[0..3] as its bytes 0..3: a 4 x 4 byte transpose in eight byte
// permutes (pairs interleaved by byte, then by byte pair).
__device__ __forceinline__ void transpose_bytes4(const uint32_t (&in)[4], uint32_t* out) {
  const uint32_t ab_lo = __byte_perm(in[0], in[1], 0x5140), ab_hi = __byte_perm(in[0], in[1], 0x7362);
  const uint32_t cd_lo = __byte_perm(in[2], in[3], 0x5140), cd_hi = __byte_perm(in[2], in[3], 0x7362);
  out[0] = __byte_perm(ab_lo, cd_lo, 0x5410);
  out[1] = __byte_perm(ab_lo, cd_lo, 0x7632);
  out[2] = __byte_perm(ab_hi, cd_hi, 0x5410);
  out[3] = __byte_perm(ab_hi, cd_hi, 0x7632);
}

// Before the wait: the thread's first norm weights, and the vector length's reciprocal.
__device__ __forceinline__ void prologue_early(const MatrowParams& p, Scratch* sc, NormWeights& nw) {
  const uint32_t n = p.cols, words = p.pitch / 4;
  const bool norm = p.pro == kProNorm;
#pragma unroll
  for (int j = 0; j < kPG; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t g = threadIdx.x + j * kThreads, i = 4 * g + e;
      nw.w[j][e] = norm && g < words && i < n ? __ldg(p.norm_w + i) : 0;
    }
  if (norm && threadIdx.x == (p.ss_in ? 0 : 32)) sc->divn = make_invdiv_fast(n);
}

// Packs the input vector (optionally residual-added and RMS-normalised) into byte planes.
// Returns the wrapping sum of the vector in *S and the limb count.
__device__ int prologue(const MatrowParams& p, uint32_t* planes32, Scratch* sc,
                        unsigned long long* S_out, const NormWeights& nw, bool running) {
  const uint32_t n = p.cols, words = p.pitch / 4;
  const bool norm = p.pro == kProNorm;
  const bool held = words <= (uint32_t)kPG * kThreads;  // one batch: values stay in registers
  int64_t xv[kPG][4];
  if (!norm && p.in_planes) {
    // the producer wrote the planes: copy the first four into shared memory while the
    // partial sums and ORs are added up, then the rest if the vector needs more limbs
    const uint32_t pbytes = p.pitch;  // bytes of one plane
    for (uint32_t k = 0; k < 4; ++k)
      for (uint32_t o = 16 * threadIdx.x; o < pbytes; o += 16 * kThreads)
        cp_async16(reinterpret_cast<uint8_t*>(planes32) + (size_t)k * pbytes + o, p.in_planes + (size_t)k * pbytes + o);
    unsigned long long S = 0, orv = 0;
    for (uint32_t i = threadIdx.x; i < p.nparts; i += kThreads) {
      S += p.parts_in[2 * i];
      orv |= p.parts_in[2 * i + 1];
    }
    block_sum_or(S, orv, sc);
    int L = 1;
    while (L < 8 && (orv >> (8 * L - 1)) != 0) ++L;
    for (uint32_t k = 4; k < (uint32_t)L; ++k)
      for (uint32_t o = 16 * threadIdx.x; o < pbytes; o += 16 * kThreads)
        cp_async16(reinterpret_cast<uint8_t*>(planes32) + (size_t)k * pbytes + o, p.in_planes + (size_t)k * pbytes + o);
    cp_async_wait_all();
    __syncthreads();
    *S_out = S;
    return L;
  }
  if (norm && p.ss_in) {
    // the producer added up the squares: the values load while thread 0 forms the RMS
    // reciprocal, then one pass normalises and packs
    if (held) {
#pragma unroll
      for (int j = 0; j < kPG; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t g = threadIdx.x + j * kThreads, i = 4 * g + e;
          xv[j][e] = g < words && i < n ? p.in[i] : 0;
        }
    }
    if (threadIdx.x == 0) {
      const unsigned long long ss = *reinterpret_cast<const volatile unsigned long long*>(p.ss_in);
      uint64_t rms = isqrt_u64(udiv_inv(ss, sc->divn) + 42950ull);  // floor(ss / n)
      if (rms < 1) rms = 1;
      sc->div = make_invdiv_fast((uint32_t)rms);
    }
    __syncthreads();
  } else if (norm) {
    // "RMS normalization": rms = isqrt(sum(x*x) / n + 42,950), at least 1.
    unsigned long long ss = 0, dummy = 0;
    for (uint32_t g0 = threadIdx.x; g0 < words; g0 += kPG * kThreads) {
#pragma unroll
      for (int j = 0; j < kPG; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t g = g0 + j * kThreads, i = 4 * g + e;
          xv[j][e] = g < words && i < n ? load_x(p, i) : 0;
        }
#pragma unroll
      for (int j = 0; j < kPG; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t g = g0 + j * kThreads, i = 4 * g + e;
          if (running && g < words && i < n && p.res_out && blockIdx.x == 0) p.res_out[i] = xv[j][e];
          ss += (unsigned long long)xv[j][e] * (unsigned long long)xv[j][e];
        }
    }
    block_sum_or(ss, dummy, sc);
    if (threadIdx.x == 0) {
      uint64_t rms = isqrt_u64(udiv_inv(ss, sc->divn) + 42950ull);  // floor(ss / n)
      if (rms < 1) rms = 1;
      sc->div = make_invdiv_fast((uint32_t)rms);
    }
    __syncthreads();
  }
  unsigned long long S = 0, orv = 0;
  if (!norm) {
    // plain: kPGP groups a thread load at once
    for (uint32_t g0 = threadIdx.x; g0 < words; g0 += kPGP * kThreads) {
      int64_t pv[kPGP][4];
#pragma unroll
      for (int j = 0; j < kPGP; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t g = g0 + j * kThreads, i = 4 * g + e;
          pv[j][e] = g < words && i < n ? (p.in_acc ? (int64_t)p.in_acc[i] >> 24 : p.in[i]) : 0;
        }
#pragma unroll
      for (int j = 0; j < kPGP; ++j) {
        const uint32_t g = g0 + j * kThreads;
        if (g >= words) break;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          // the shifted attention outputs, kept in the state by block 0
          if (p.in_acc && running && blockIdx.x == 0 && 4 * g + e < n) p.in_out[4 * g + e] = pv[j][e];
          S += (unsigned long long)pv[j][e];
          orv |= (unsigned long long)(pv[j][e] ^ (pv[j][e] >> 63));
        }
        const uint32_t lo[4] = {(uint32_t)pv[j][0], (uint32_t)pv[j][1], (uint32_t)pv[j][2], (uint32_t)pv[j][3]};
        const uint32_t hi[4] = {(uint32_t)((uint64_t)pv[j][0] >> 32), (uint32_t)((uint64_t)pv[j][1] >> 32),
                                (uint32_t)((uint64_t)pv[j][2] >> 32), (uint32_t)((uint64_t)pv[j][3] >> 32)};
        uint32_t pl[8];
        transpose_bytes4(lo, pl);
        transpose_bytes4(hi, pl + 4);
#pragma unroll
        for (int k = 0; k < 8; ++k) planes32[k * words + g] = pl[k];
      }
    }
  }
  const InvDiv D = sc->div;
  for (uint32_t g0 = threadIdx.x; norm && g0 < words; g0 += kPG * kThreads) {
    int32_t wv[kPG][4];
#pragma unroll
    for (int j = 0; j < kPG; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t g = g0 + j * kThreads, i = 4 * g + e;
        const bool ok = g < words && i < n;
        if (!(norm && held)) xv[j][e] = ok ? (norm ? load_x(p, i) : p.in[i]) : 0;
        wv[j][e] = !norm ? 0 : held ? nw.w[j][e] : ok ? __ldg(p.norm_w + i) : 0;
      }
#pragma unroll
    for (int j = 0; j < kPG; ++j) {
      const uint32_t g = g0 + j * kThreads;
      if (g >= words) break;
      int64_t v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // norm: y = ((x * w) / rms) >> 8, the division truncating toward zero
        const int64_t val = norm ? sdiv_trunc(wmul(xv[j][e], (int64_t)wv[j][e]), D) >> 8 : xv[j][e];
        v[e] = val;
        S += (unsigned long long)val;
        orv |= (unsigned long long)(val ^ (val >> 63));
      }
      // plane k's word g holds byte k of the four values: a 4 x 4 byte transpose of their
      // low and of their high halves
      const uint32_t lo[4] = {(uint32_t)v[0], (uint32_t)v[1], (uint32_t)v[2], (uint32_t)v[3]};
      const uint32_t hi[4] = {(uint32_t)((uint64_t)v[0] >> 32), (uint32_t)((uint64_t)v[1] >> 32),
                              (uint32_t)((uint64_t)v[2] >> 32), (uint32_t)((uint64_t)v[3] >> 32)};
      uint32_t pl[8];
      transpose_bytes4(lo, pl);
      transpose_bytes4(hi, pl + 4);
#pragma unroll
      for (int k = 0; k < 8; ++k) planes32[k * words + g] = pl[k];
    }
  }
  block_sum_or(S, orv, sc);
  int L = 1;
  while (L < 8 && (orv >> (8 * L - 1)) != 0) ++L;
  *S_out = S;
  return L;
}

// Epilogue of one finished row: y is its scaled sum, partner that of row ^ 1 (the other half
// of a gate/up or rotary pair; unused for plain stores).
__device__ __forceinline__ void epilogue(const MatrowParams& p, uint32_t row, int64_t y,
                                         int64_t partner, uint32_t pos) {
  if (p.epi == kEpiStore) {
    p.out[row] = y;
  } else if (p.epi == kEpiSiLU) {
    // rows 2j (gate) and 2j+1 (up): h_j = (silu(g) * u) >> 16
    if ((row & 1) == 0) p.out[row >> 1] = wmul(silu_lookup(y, p.silu_tab), partner) >> 16;
  } else {  // kEpiQKV
    const bool even = (row & 1) == 0;
    const int64_t a = even ? y : partner, b = even ? partner : y;
    if (row < p.q_rows) {
      const uint32_t j = (row % p.head_dim) >> 1;
      const int32_t* cs = p.rope + ((size_t)pos * (p.head_dim >> 1) + j) * 2;
      int64_t a2, b2;
      rotate_pair(a, b, __ldg(cs), __ldg(cs + 1), a2, b2);
      p.out[row] = even ? a2 : b2;
    } else if (row < p.q_rows + p.kv_dim) {
      const uint32_t e = row - p.q_rows;
      if (!fits_i32(y)) record_error(p.state, err_key(pos, p.layer, 6, e));
      const uint32_t j = (e % p.head_dim) >> 1;
      const int32_t* cs = p.rope + ((size_t)pos * (p.head_dim >> 1) + j) * 2;
      int64_t a2, b2;
      rotate_pair((int64_t)(int32_t)a, (int64_t)(int32_t)b, __ldg(cs), __ldg(cs + 1), a2, b2);
      const int64_t mine = even ? a2 : b2;
      if (!fits_i32(mine)) record_error(p.state, err_key(pos, p.layer, 8, e));
      p.kcache[cache_word(e, pos, p.head_dim, p.cache)] = (int32_t)mine;
    } else {
      const uint32_t e = row - p.q_rows - p.kv_dim;
      if (!fits_i32(y)) record_error(p.state, err_key(pos, p.layer, 7, e));
      p.vcache[cache_word(e, pos, p.head_dim, p.cache)] = (int32_t)y;
    }
  }
}

// The rows of a CTA: an even-aligned share of the row pairs, so that both rows of a gate/up
// or rotary pair finish in the same CTA.
__device__ __forceinline__ void cta_rows(const MatrowParams& p, uint32_t& rb, uint32_t& re) {
  const uint32_t pairs = (p.rows + 1) / 2;
  rb = 2 * (uint32_t)((uint64_t)blockIdx.x * pairs / gridDim.x);
  re = min(2 * (uint32_t)((uint64_t)(blockIdx.x + 1) * pairs / gridDim.x), p.rows);
}

// Loads work item `it` of the chunk [c0, c1) into w: rows c0 + kG * (it / ns) onwards (at
// most kG, not past c1) over the 512-byte column slice it % ns, 16 bytes a lane.  Rows past the
// chunk, columns past the pitch and items past the last read as zero bytes.
template <bool kGrouped>
__device__ __forceinline__ void load_item(const MatrowParams& p, uint32_t c0, uint32_t c1,
                                          uint32_t ns, uint32_t it, uint32_t items, uint4 (&w)[kG]) {
  const int lane = threadIdx.x & 31;
  const uint32_t g = it / ns, s = it - g * ns;
  const uint32_t r0 = c0 + g * kG, c = s * kSlice + lane * 16;
  const bool live = it < items && c < p.pitch;
  const size_t gstride = (size_t)p.rows * kGroupCols;  // grouped: bytes between column groups
#pragma unroll
  for (int r = 0; r < kG; ++r) {
    const uint32_t row = r0 + r;
    w[r] = make_uint4(0u, 0u, 0u, 0u);
    if (live && row < c1) {
      w[r] = kGrouped ? ld_stream16(p.W + (size_t)row * kGroupCols + (size_t)(c >> 7) * gstride +
                                    ((c & 0x70u) ^ ((row & 7u) << 4)))
                      : ld_stream16(p.W + (size_t)row * p.pitch + c);
    }
  }
}

// Sums the eight per-lane values v[0..7] over the warp: afterwards every lane holds the
// total of row (lane >> 2).  Each exchange step halves the values a lane carries, so the
// whole reduction takes nine 64-bit shuffles instead of eight full butterflies.
__device__ __forceinline__ unsigned long long reduce_rows8(const unsigned long long (&v)[kG]) {
  const int lane = threadIdx.x & 31;
  unsigned long long u[4], t[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const unsigned long long keep = b4 ? v[j + 4] : v[j], send = b4 ? v[j] : v[j + 4];
    u[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const unsigned long long keep = b3 ? u[j + 2] : u[j], send = b3 ? u[j] : u[j + 2];
    t[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  unsigned long long s = (b2 ? t[1] : t[0]) + __shfl_xor_sync(0xffffffffu, b2 ? t[0] : t[1], 4);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  return s;
}

// Accumulates rows [h, h + H) of an item: byte-plane dp4a runs, then each row's planes
// recombined into one 64-bit partial (the top plane signed).
template <int L, int H>
__device__ __forceinline__ void item_rows(const uint4 (&w)[kG], const uint8_t* xp, uint32_t pitch,
                                          int h, unsigned long long (&sums)[kG]) {
  uint32_t acc[H][L];
#pragma unroll
  for (int r = 0; r < H; ++r)
#pragma unroll
    for (int k = 0; k < L; ++k) acc[r][k] = 0;
#pragma unroll
  for (int k = 0; k < L; ++k) {
    const uint4 xk = *reinterpret_cast<const uint4*>(xp + (size_t)k * pitch);
#pragma unroll
    for (int r = 0; r < H; ++r) {
      const uint4 wr = w[h + r];
      if (k < L - 1) {
        uint32_t a = acc[r][k];
        a = __dp4a(wr.x, xk.x, a);
        a = __dp4a(wr.y, xk.y, a);
        a = __dp4a(wr.z, xk.z, a);
        a = __dp4a(wr.w, xk.w, a);
        acc[r][k] = a;
      } else {
        int a = (int)acc[r][k];
        a = dp4a_us(wr.x, xk.x, a);
        a = dp4a_us(wr.y, xk.y, a);
        a = dp4a_us(wr.z, xk.z, a);
        a = dp4a_us(wr.w, xk.w, a);
        acc[r][k] = (uint32_t)a;
      }
    }
  }
#pragma unroll
  for (int r = 0; r < H; ++r) {
    unsigned long long a = 0;
#pragma unroll
    for (int k = 0; k < L; ++k) {
      const unsigned long long t = (k < L - 1) ? (unsigned long long)acc[r][k]
                                               : (unsigned long long)(long long)(int)acc[r][k];
      a += t << (8 * k);
    }
    sums[h + r] = a;
  }
}

// Rows [rb, re) of W, in chunks of at most kChunkRows.  A chunk's work items (kG rows by one
// 512-byte slice) go round-robin to the warps, each warp loading its next item while it works
// on the current one; each item's per-row partials add into the chunk's row totals in shared
// memory, and once all items are in, one thread per row applies the -128 * sum(x) correction,
// the row scale and the epilogue.  wn holds the warp's first item of the first chunk, loaded
// before the vector was packed.
// Rows of W: row-major with the given pitch, or (kGrouped) the model's column-group layout,
// where the 16-byte chunk at column c of row r sits at grouped_offset(rows, r, c).
template <int L, bool kGrouped>
__device__ void rows_loop(const MatrowParams& p, const uint8_t* planes, Scratch* sc,
                          unsigned long long S, uint32_t pos, uint32_t rb, uint32_t re,
                          uint4 (&wn)[kG]) {
  constexpr int H = L <= 4 ? kG / 2 : kG / 4;  // rows accumulated at once (register budget)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t pitch = p.pitch, ns = (pitch + kSlice - 1) / kSlice;
  unsigned long long hs = 0, ho = 0;  // the CTA's SiLU outputs: wrapping sum, OR of |h|
  for (uint32_t c0 = rb; c0 < re; c0 += kChunkRows) {
    const uint32_t c1 = min(c0 + kChunkRows, re);
    const uint32_t items = (c1 - c0 + kG - 1) / kG * ns;
    if (c0 != rb) load_item<kGrouped>(p, c0, c1, ns, warp, items, wn);
    // the finishing thread's row scales, fetched while the items stream
    const uint32_t frow = c0 + threadIdx.x, fprow = frow ^ 1u;
    const uint32_t fscale = frow < c1 ? __ldg(p.scale + frow) : 0u;
    const uint32_t fpscale = frow < c1 && fprow < c1 ? __ldg(p.scale + fprow) : 0u;
    // the residual inputs of the chunk's rows, copied into shared memory while the items stream
    if (p.resid_out && frow < c1) cp_async8(&sc->res[threadIdx.x], p.resid_in + frow);
    for (uint32_t it = warp; it < items; it += kWarps) {
      uint4 w[kG];
#pragma unroll
      for (int r = 0; r < kG; ++r) w[r] = wn[r];
      load_item<kGrouped>(p, c0, c1, ns, it + kWarps, items, wn);
      const uint32_t g = it / ns, s = it - g * ns;
      const uint32_t r0 = c0 + g * kG;
      const uint32_t c = s * kSlice + lane * 16;
      unsigned long long sums[kG];
      if (c < pitch) {
        const uint8_t* xp = planes + c;
#pragma unroll
        for (int h = 0; h < kG; h += H) item_rows<L, H>(w, xp, pitch, h, sums);
      } else {
#pragma unroll
        for (int r = 0; r < kG; ++r) sums[r] = 0;
      }
      const unsigned long long tot = reduce_rows8(sums);
      const uint32_t rl = r0 - c0 + (uint32_t)(lane >> 2);
      if ((lane & 3) == 0 && c0 + rl < c1) atomicAdd(&sc->tot[rl], tot);
    }
    if (p.resid_out) cp_async_wait_all();
    __syncthreads();
    unsigned long long sq = 0;
    if (frow < c1) {
      const uint32_t t = threadIdx.x;
      const int64_t y = (int64_t)((sc->tot[t] - (S << 7)) * (unsigned long long)fscale) >> 24;
      const int64_t partner =
          fprow < c1 ? (int64_t)((sc->tot[t ^ 1u] - (S << 7)) * (unsigned long long)fpscale) >> 24 : 0;
      epilogue(p, frow, y, partner, pos);
      if (p.planes_out && (frow & 1u) == 0) {
        // the SiLU output h_j (as the epilogue stored it) as byte planes for the next kernel
        const int64_t hv = wmul(silu_lookup(y, p.silu_tab), partner) >> 16;
        const uint32_t j = frow >> 1;
#pragma unroll
        for (int k = 0; k < 8; ++k) p.planes_out[(size_t)k * p.planes_pitch + j] = (uint8_t)((uint64_t)hv >> (8 * k));
        hs += (unsigned long long)hv;
        ho |= (unsigned long long)(hv ^ (hv >> 63));
      }
      if (p.resid_out) {
        // the residual (phases 11 and 16) and its square for the next normalization
        const int64_t xr = wadd(sc->res[t], y);
        p.resid_out[frow] = xr;
        sq = (unsigned long long)xr * (unsigned long long)xr;
      }
    }
    if (p.resid_out && (threadIdx.x & ~31u) < c1 - c0) {
      sq = warp_sum(sq);
      if ((threadIdx.x & 31) == 0) atomicAdd(p.ss_out, sq);
    }
    __syncthreads();
    for (uint32_t t = threadIdx.x; t < kChunkRows; t += kThreads) sc->tot[t] = 0;
    __syncthreads();
  }
  if (p.planes_out) {
    block_sum_or(hs, ho, sc);
    if (threadIdx.x == 0) {
      p.parts_out[2 * blockIdx.x] = hs;
      p.parts_out[2 * blockIdx.x + 1] = ho;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) k_matrow(const MatrowParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t rb, re;
  cta_rows(p, rb, re);
  // The warp's first weights are requested before anything else: weights are never written,
  // so this may run while the previous kernel on the stream is still finishing (the launch
  // allows programmatic dependent launch).  Everything that reads what earlier kernels wrote
  // (the state header, the vector) waits for their completion first.
  uint4 wn[kG];
  if (rb < re) {
    const uint32_t ns = (p.pitch + kSlice - 1) / kSlice, c1 = min(rb + kChunkRows, re);
    const uint32_t items = (c1 - rb + kG - 1) / kG * ns;
    if (p.grouped)
      load_item<true>(p, rb, c1, ns, threadIdx.x >> 5, items, wn);
    else
      load_item<false>(p, rb, c1, ns, threadIdx.x >> 5, items, wn);
  }
  uint8_t* planes = smem;
  Scratch* sc = reinterpret_cast<Scratch*>(smem + 8 * (size_t)p.pitch);
  NormWeights nw;
  prologue_early(p, sc, nw);
  wait_prior_grids();
  allow_next_grid();
  if (p.acc_clear) {  // the previous kernel has read these sums: clear them for their next use
    const uint32_t w0 = (uint32_t)((uint64_t)blockIdx.x * p.acc_words / gridDim.x);
    const uint32_t w1 = (uint32_t)((uint64_t)(blockIdx.x + 1) * p.acc_words / gridDim.x);
    for (uint32_t i = w0 + threadIdx.x; i < w1; i += kThreads) p.acc_clear[i] = 0;
  }
  if (rb >= re) return;
  // The state's phase is read here but tested only after the prologue, so that its vector
  // loads need not wait for it: for a failed state the prologue skips its one kind of global
  // store (the residual copy) and the kernel returns after it.  Every thread reads the same
  // header word, which nothing writes while this kernel runs.
  const bool running = !p.state || hdr_ld<uint32_t>(p.state, kHPhase) == CK_PHASE_RUNNING;
  const uint32_t pos = p.state ? hdr_ld<uint32_t>(p.state, kHPosition) : 0u;
  for (uint32_t t = threadIdx.x; t < kChunkRows; t += kThreads) sc->tot[t] = 0;
  unsigned long long S;
  const int L = prologue(p, reinterpret_cast<uint32_t*>(planes), sc, &S, nw, running);
  if (!running) return;
  if (p.grouped) {
    switch (L) {
      case 1: rows_loop<1, true>(p, planes, sc, S, pos, rb, re, wn); break;
      case 2: rows_loop<2, true>(p, planes, sc, S, pos, rb, re, wn); break;
      case 3: rows_loop<3, true>(p, planes, sc, S, pos, rb, re, wn); break;
      case 4: rows_loop<4, true>(p, planes, sc, S, pos, rb, re, wn); break;
      case 5: rows_loop<5, true>(p, planes, sc, S, pos, rb, re, wn); break;
      case 6: rows_loop<6, true>(p, planes, sc, S, pos, rb, re, wn); break;
      case 7: rows_loop<7, true>(p, planes, sc, S, pos, rb, re, wn); break;
      default: rows_loop<8, true>(p, planes, sc, S, pos, rb, re, wn); break;
    }
  } else {
    switch (L) {
      case 1: rows_loop<1, false>(p, planes, sc, S, pos, rb, re, wn); break;
      case 2: rows_loop<2, false>(p, planes, sc, S, pos, rb, re, wn); break;
      case 3: rows_loop<3, false>(p, planes, sc, S, pos, rb, re, wn); break;
      case 4: rows_loop<4, false>(p, planes, sc, S, pos, rb, re, wn); break;
      case 5: rows_loop<5, false>(p, planes, sc, S, pos, rb, re, wn); break;
      case 6: rows_loop<6, false>(p, planes, sc, S, pos, rb, re, wn); break;
      case 7: rows_loop<7, false>(p, planes, sc, S, pos, rb, re, wn); break;
      default: rows_loop<8, false>(p, planes, sc, S, pos, rb, re, wn); break;
    }
  }
}

}  // namespace

size_t matrow_smem_bytes(uint32_t pitch) { return 8 * (size_t)pitch + sizeof(Scratch); }

cudaError_t configure_matrow() {
  return cudaFuncSetAttribute(k_matrow, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)matrow_smem_bytes(16384));
}

cudaError_t launch_matrow(const MatrowParams& p, cudaStream_t s, int num_sms) {
  const size_t smem = matrow_smem_bytes(p.pitch);
  if (p.pitch > 16384) return cudaErrorInvalidValue;
  const uint32_t pairs = (p.rows + 1) / 2;
  uint32_t blocks = pairs < (uint32_t)num_sms ? pairs : (uint32_t)num_sms;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_matrow, p);
}

}  // namespace ck
