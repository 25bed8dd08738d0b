// Layer-major prefill: the prompt positions of one run go through each layer together
// ("The inference core", "The forward pass, in order": phases 3 to 16 for every position
// that generates no token).
//
// Position by position, every matrix is read from memory once per position.  Here a chunk
// of P prompt positions moves through a layer at once, so each matrix is read once per
// chunk and its matrix rows ("A matrix row") for all P positions become one dense
// contraction  Y[n][r] = sum_c (byte[r][c] - 128) * x[n][c]  on the tensor cores.
//
// Exactness.  When every x of a vector fits 8L signed bits,
//   x = sum_{k<L-1} 256^k u_k + 256^(L-1) s,   u_k bytes (0..255), s a signed byte,
// so the contraction splits into L contractions over byte planes.  Every plane value and
// every (byte - 128) is an integer of at most 8 bits, exact in f16; the warp MMA forms the
// products exactly and adds them in f32, which is exact while every partial sum stays
// below 2^24: 512 columns of |(byte - 128) u| <= 128 * 255 = 32,640 reach at most
// 16,711,680.  So every 512 columns the f32 sums move into i32 accumulators (whole rows stay
// below 2^31 up to 65,793 columns), and the planes are combined modulo 2^64 with the row
// scale and the >> 24: the same bits as the wrapping definition, since
// sum_c byte*x - 128 * sum_c x = sum_c (byte - 128) x  modulo 2^64.
//
// The rest of each layer (normalization, rotary, checked cache stores, attention over the
// run's cache with the causal limit of each position, SiLU gating, residuals) runs per
// position exactly as in the one-position kernels, P positions per launch.  A cache store
// that does not fit records the smallest (position, layer, phase, element) key, which is the
// first failing store in position order, since no position reads a later position's values.
#include <cuda_fp16.h>

#include "ck_internal.cuh"

namespace ck {
namespace {

constexpr uint32_t kBM = 128;        // contraction tile: 128 matrix rows
constexpr uint32_t kBN = 64;         // x 64 plane columns (positions of one plane)
constexpr uint32_t kBK = 128;        // x 128 columns, one column group
constexpr uint32_t kBTile = kBN * kBK * 2;   // f16 planes: one 64 x 128 tile
constexpr uint32_t kFlushGroups = 4;         // column groups between f32 -> i32 moves
constexpr int kRowThreads = 256;

enum BEpi : int { kBEpiQKV = 0, kBEpiResid = 1, kBEpiSiLU = 2, kBEpiLogits = 3 };

// A chunk of one run is gated by that run's state: a position earlier in the same turn
// that failed it stops the chunk.  A batch of runs has no gate (nullptr).
__device__ __forceinline__ bool running(const uint8_t* gate) {
  return gate == nullptr || hdr_ld<uint32_t>(gate, kHPhase) == CK_PHASE_RUNNING;
}

// Programmatic dependent launch: the per-layer kernels are launched so that their blocks may
// be scheduled while the previous kernel on the stream finishes; each waits here, before its
// first global read or write, until that kernel has completed and its writes are visible.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ int32_t* layer_cache(const RowDesc& r, uint64_t off, uint32_t layer,
                                                uint32_t kv_dim) {
  return reinterpret_cast<int32_t*>(r.st + off) + (size_t)layer * r.cache * kv_dim;
}

// Limbs of a vector from the OR of x ^ (x >> 63) over it: the smallest L with every x in
// 8L signed bits.
__device__ __forceinline__ int limbs_of_or(unsigned long long orv) {
  int L = 1;
  while (L < 8 && (orv >> (8 * L - 1)) != 0) ++L;
  return L;
}

__device__ __forceinline__ unsigned long long bwarp_sum(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ unsigned long long bwarp_or(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block-wide sum (every thread gets it); red holds blockDim.x / 32 words.
__device__ unsigned long long block_sum(unsigned long long v, unsigned long long* red) {
  v = bwarp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (uint32_t w = 0; w < blockDim.x / 32; ++w) t += red[w];
  __syncthreads();
  return t;
}

// One atomic OR per block of the values' x ^ (x >> 63).
__device__ void block_or_to(unsigned long long v, unsigned long long* dst, unsigned long long* red) {
  v = bwarp_or(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t = 0;
    for (uint32_t w = 0; w < blockDim.x / 32; ++w) t |= red[w];
    if (t) atomicOr(dst, t);
  }
}

// ------------------------------------------------------------------ phase 3 and norms

// Phase 3 for every row (one block each): the row's token is its run's prompt id at the
// position, or the token generated there; x = ((byte - 128) * scale) >> 8.
__global__ void __launch_bounds__(kRowThreads) k_bembed(const uint8_t* gate, const RowDesc* rows,
                                                         int64_t* X, uint32_t d, const uint8_t* E,
                                                         const uint32_t* Es, uint32_t vocab,
                                                         int32_t* rstat) {
  if (!running(gate)) return;
  const uint32_t n = blockIdx.x;
  const RowDesc r = rows[n];
  const uint32_t tok = r.pos < r.np ? reinterpret_cast<const uint32_t*>(r.st + r.off_prompt)[r.pos]
                                    : reinterpret_cast<const uint32_t*>(r.st + r.off_out)[r.pos - r.np];
  int64_t* x = X + (size_t)n * d;
  if (tok >= vocab) {  // a state edited outside the library: that position fails
    if (threadIdx.x == 0) rstat[n] = CK_INVALID_STATE;
    for (uint32_t i = threadIdx.x; i < d; i += blockDim.x) x[i] = 0;
    return;
  }
  const int64_t s = (int64_t)__ldg(Es + tok);
  for (uint32_t i = threadIdx.x; i < d; i += blockDim.x)
    x[i] = ((int64_t)E[grouped_offset(vocab, tok, i)] - 128) * s >> 8;
}

// "RMS normalization" of each position's row (one block each): rms = max(isqrt(sum x^2 / d
// + 42,950), 1), y = ((x * w) / rms) >> 8 with the division truncating; ORs the outputs'
// magnitudes into *orw for the plane count.  A block of kNormThreads: a row's loads go out
// at once (the kernel is a chain of dependent steps over a few rows).  The first kNormPer
// elements a thread stay in registers between the two passes, their norm weights are loaded
// before the wait (model data), and both divisions by invariant divisors (d, then rms) use
// reciprocals built from single-precision estimates with exact corrections.
constexpr int kNormThreads = 1024;
constexpr int kNormPer = 4;  // elements a thread keeps (rows up to 4,096)
__global__ void __launch_bounds__(kNormThreads) k_bnorm(const uint8_t* gate, const int64_t* X,
                                                         int64_t* XB, const int32_t* w, uint32_t d,
                                                         unsigned long long* orw) {
  __shared__ unsigned long long red[kNormThreads / 32];
  __shared__ InvDiv div;
  int32_t wv[kNormPer];
#pragma unroll
  for (int j = 0; j < kNormPer; ++j) {
    const uint32_t i = threadIdx.x + j * kNormThreads;
    wv[j] = i < d ? __ldg(w + i) : 0;
  }
  const InvDiv Dd = make_invdiv_fast(d);  // floor(ss / d) by a multiply
  pdl_enter();
  if (!running(gate)) return;
  const int64_t* x = X + (size_t)blockIdx.x * d;
  int64_t* y = XB + (size_t)blockIdx.x * d;
  int64_t xv[kNormPer];
  unsigned long long ss = 0;
#pragma unroll
  for (int j = 0; j < kNormPer; ++j) {
    const uint32_t i = threadIdx.x + j * kNormThreads;
    xv[j] = i < d ? x[i] : 0;
    ss += (unsigned long long)xv[j] * (unsigned long long)xv[j];
  }
  for (uint32_t i = threadIdx.x + kNormPer * kNormThreads; i < d; i += kNormThreads)
    ss += (unsigned long long)x[i] * (unsigned long long)x[i];
  ss = block_sum(ss, red);
  if (threadIdx.x == 0) {
    uint64_t rms = isqrt_u64(udiv_inv(ss, Dd) + 42950ull);
    if (rms < 1) rms = 1;
    div = make_invdiv_fast((uint32_t)rms);
  }
  __syncthreads();
  const InvDiv D = div;
  unsigned long long o = 0;
#pragma unroll
  for (int j = 0; j < kNormPer; ++j) {
    const uint32_t i = threadIdx.x + j * kNormThreads;
    if (i < d) {
      const int64_t v = sdiv_trunc(wmul(xv[j], (int64_t)wv[j]), D) >> 8;
      y[i] = v;
      o |= (unsigned long long)(v ^ (v >> 63));
    }
  }
  for (uint32_t i = threadIdx.x + kNormPer * kNormThreads; i < d; i += kNormThreads) {
    const int64_t v = sdiv_trunc(wmul(x[i], (int64_t)__ldg(w + i)), D) >> 8;
    y[i] = v;
    o |= (unsigned long long)(v ^ (v >> 63));
  }
  block_or_to(o, orw, red);
}

// ------------------------------------------------------------------ byte planes

// Plane layout, read by the contraction one 16 KB tile at a time: plane column
// n' = k * Npad + n (plane k of position n), tiles of 64 plane columns x 128 columns stored
// tile after tile (column groups inner).  A tile is the MMA's K-major operand layout with the
// 128-byte swizzle: two atom columns of 64 columns each (64 rows of 128 bytes), the 16-byte
// chunk c of row i at c ^ (i & 7).
__device__ __forceinline__ uint64_t plane_offset(uint32_t np, uint32_t KG, uint32_t kg, uint32_t chunk) {
  const uint32_t nt = np / kBN, nl = np % kBN;
  return ((uint64_t)nt * KG + kg) * kBTile + (chunk >> 3) * (kBN * 128) + (uint64_t)nl * 128 +
         (((chunk & 7u) ^ (nl & 7u)) << 4);
}

// Writes planes 0 .. L-1 of the P vectors V (row stride ld, cols used), zero beyond P and
// cols.  One thread per 8 columns of one position: it loads the 8 values once and writes
// their L planes.  With clear_rows > 0 it also zeroes the next contraction's output S[n'][r]
// (n' < L * Npad, r < clear_rows), which a contraction split over column ranges adds into.
__global__ void __launch_bounds__(kRowThreads) k_bplanes(const uint8_t* gate, const int64_t* V,
                                                          uint32_t ld, uint32_t P, uint32_t cols,
                                                          uint32_t Npad, uint32_t KG,
                                                          const unsigned long long* orw, uint8_t* B,
                                                          int32_t* S, uint32_t clear_rows) {
  pdl_enter();
  if (!running(gate)) return;
  const int L = limbs_of_or(*orw);
  if (clear_rows) {
    const uint64_t words = (uint64_t)L * Npad * clear_rows;
    for (uint64_t q = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; q < words;
         q += (uint64_t)gridDim.x * blockDim.x)
      S[q] = 0;
  }
  const uint32_t per_row = KG * 16;  // 8-column chunks of a row
  const uint32_t total = Npad * per_row;
  for (uint32_t q = blockIdx.x * blockDim.x + threadIdx.x; q < total; q += gridDim.x * blockDim.x) {
    const uint32_t n = q / per_row, cc = q - n * per_row;
    const uint32_t kg = cc >> 4, ch = cc & 15u, c0 = kg * kBK + ch * 8;
    int64_t xv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t c = c0 + e;
      xv[e] = (n < P && c < cols) ? V[(size_t)n * ld + c] : 0;
    }
    for (int k = 0; k < L; ++k) {
      uint32_t h[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        int v2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u)
          v2[u] = (k + 1 < L) ? (int)(((uint64_t)xv[e + u] >> (8 * k)) & 0xFFu)
                              : (int)(xv[e + u] >> (8 * k));  // top plane: signed
        const __half2 hv = __halves2half2(__int2half_rn(v2[0]), __int2half_rn(v2[1]));
        h[e >> 1] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      *reinterpret_cast<uint4*>(B + plane_offset(k * Npad + n, KG, kg, ch)) = make_uint4(h[0], h[1], h[2], h[3]);
    }
  }
}

// ------------------------------------------------------------------ the contraction

// The 5th-generation tensor cores (tcgen05): one thread issues 128 x N x 16 MMAs whose f32
// accumulators live in tensor memory (TMEM); A (the weights widened to f16) is read from
// tensor memory, B (the planes) from shared memory through a matrix descriptor: K-major with
// the 128-byte swizzle, 8-row atoms of 128-byte rows, row r's 16-byte chunk j at j ^ (r & 7),
// atoms 1,024 bytes apart.  The weights' column-group layout is that pattern for bytes, so
// a weight tile arrives with one bulk copy and each row is found at a fixed place to widen;
// the planes are stored in the pattern as f16.
constexpr uint32_t kTN = 192;                  // most plane columns per block (three planes of 64)
constexpr uint32_t kTcConvWarps = 8;           // widen the weights, drain the accumulators
constexpr int kTcThreads = 32 * (kTcConvWarps + 2);  // + a producer warp and an MMA warp
constexpr uint32_t kRing = 4;                  // weight-byte and plane stages in flight (tiles up to
                                               // 128 plane columns; 3 for wider ones)
constexpr uint32_t kAu8 = kBM * kBK;           // 16 KB: 128 rows x 128 weight bytes
__host__ __device__ constexpr uint32_t ring_of(uint32_t n) { return n > 128 ? 3u : kRing; }
__host__ __device__ constexpr uint32_t tile_smem(uint32_t n) {  // ring of weight bytes and planes
  return ring_of(n) * (kAu8 + 2 * n * 128);
}
constexpr uint32_t kTcSmem = (tile_smem(128) > tile_smem(kTN) ? tile_smem(128) : tile_smem(kTN)) + 1024;
// Tensor memory (512 columns of 128 lanes): two accumulator buffers of up to kTN columns at
// columns 0 and 256, and the widened weights of two stages (128 rows x 128 f16, 64 columns
// each: lane = row, two consecutive columns' values a 32-bit column) in the gaps after them.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;             // columns between the two accumulator buffers
constexpr uint32_t kAColA = kTN, kAColB = kAccCols + kTN;  // the two weight buffers
static_assert(kTN + 64 <= kAccCols && kAccCols + kTN + 64 <= kTmemCols, "tensor memory layout");
constexpr uint32_t kTcPoll = 1u << 22;         // bounded waits

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mb_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mb_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes)
               : "memory");
}
// Adds to the transaction bytes the current phase waits for, without an arrival.
__device__ __forceinline__ void mb_expect_only(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mb_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_addr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity; gives up after kTcPoll polls, raising *abort.
__device__ __forceinline__ void mb_wait(uint64_t* b, uint32_t parity, volatile int* abort) {
  for (uint32_t it = 0; it < kTcPoll; ++it) {
    if (mb_try(b, parity)) return;
    if (*abort) return;
  }
  *abort = 1;
}
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

struct TcBars {
  uint64_t full[kRing];     // stage landed (bulk copies)
  uint64_t empty[kRing];    // stage's MMAs done: the slot may be refilled
  uint64_t conv[2];         // f16 weights of the stage in tensor memory (one arrival per converter warp)
  uint64_t f16free[2];      // MMAs reading an f16 weight buffer done
  uint64_t accf[2];         // accumulator group complete
  uint64_t accfree[2];      // accumulator buffer drained (one arrival per converter warp)
};

// Shared-memory matrix descriptor: start >> 4, leading offset (unused with the swizzle) 16
// bytes, 8-row stride 1,024 bytes, descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: f16 operands, f32 accumulator, both K-major,
// N / 8 at bit 17, M / 16 at bit 24.
__host__ __device__ constexpr uint32_t mma_idesc(uint32_t n) {
  return (1u << 4) | ((n >> 3) << 17) | ((kBM >> 4) << 24);
}

// One MMA with A (the widened weights) in tensor memory and B (planes) in shared memory.
__device__ __forceinline__ void mma_f16_ts(uint32_t tmem, uint32_t ta, uint64_t db, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }"
      ::"r"(tmem), "r"(ta), "l"(db), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_addr(bar))
               : "memory");
}

// Two weight bytes (selected by sel) as an f16 pair of byte - 128: 0x64XX is the f16 value
// 1024 + XX exactly, and subtracting 1152 leaves XX - 128, also exact.
__device__ __forceinline__ uint32_t bytes_to_f16x2(uint32_t w, uint32_t sel) {
  const uint32_t h = __byte_perm(w, 0x64646464u, sel);
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
  return r;
}

// Widens a stage's weight bytes (128 rows x 128 columns, column-group layout) to f16
// (byte - 128) into tensor memory: warp w takes rows 32 (w % 4) + lane (its lane quarter) and
// columns 64 (w / 4) .. + 63, four 16-byte chunks of its row, 32 f16 pairs stored at once.
__device__ __forceinline__ void widen_to_tmem(const uint8_t* src, uint32_t ta) {
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t r = 32 * (warp & 3u) + lane, j0 = 4 * (warp >> 2);
  uint32_t v[32];
#pragma unroll
  for (uint32_t e = 0; e < 4; ++e) {
    const uint32_t j = j0 + e;
    const uint4 w = *reinterpret_cast<const uint4*>(src + r * 128 + ((j ^ (r & 7u)) << 4));
    v[8 * e + 0] = bytes_to_f16x2(w.x, 0x5140u);
    v[8 * e + 1] = bytes_to_f16x2(w.x, 0x5342u);
    v[8 * e + 2] = bytes_to_f16x2(w.y, 0x5140u);
    v[8 * e + 3] = bytes_to_f16x2(w.y, 0x5342u);
    v[8 * e + 4] = bytes_to_f16x2(w.z, 0x5140u);
    v[8 * e + 5] = bytes_to_f16x2(w.z, 0x5342u);
    v[8 * e + 6] = bytes_to_f16x2(w.w, 0x5140u);
    v[8 * e + 7] = bytes_to_f16x2(w.w, 0x5342u);
  }
  const uint32_t addr = ta + ((32 * (warp & 3u)) << 16) + 32 * (warp >> 2);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
        "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Adds the f32 sums of one accumulator buffer (this warp's 32 rows, this warpgroup's half
// of the N columns) to the integer sums.  Every sum is an integer below 2^24: exact.
template <uint32_t N>
__device__ __forceinline__ void drain(uint32_t tmem_buf, int32_t* iacc) {
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t base = tmem_buf + ((32 * (warp & 3u)) << 16) + (warp >> 2) * (N / 2);
#pragma unroll
  for (uint32_t c = 0; c < N / 2; c += 16) {
    uint32_t v[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(base + c));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) iacc[c + i] += __float2int_rn(__uint_as_float(v[i]));
  }
}

// S[n'][r] = sum_c (W[r][c] - 128) * plane[n'][c] for the block's 128 rows and N plane
// columns (N = 192, or 128 or 64 for a last tile; plane tiles from pt0 on), over its range
// of column groups (gridDim.z
// ranges add their integer sums into S, cleared beforehand).  Warp-specialised, linked by
// mbarriers only:
//   producer (warp 8)   copies stage s (a column group's weight bytes and planes) into ring
//                       slot s % R once the MMAs of stage s - R are done;
//   converters (0..7)   widen stage s's weights into the tensor-memory f16 buffer s % 2 once
//                       the MMAs of stage s - 2 are done, and drain each finished
//                       accumulator group;
//   MMA thread (warp 9) issues stage s's eight 16-column MMAs into accumulator buffer g % 2
//                       of group g (four column groups, 512 columns: every f32 partial sum
//                       stays below 2^24) once stage s is widened and group g - 2 drained.
template <uint32_t N>
__device__ void bgemm_tile(const uint8_t* W, uint32_t rows, uint32_t KG, const uint8_t* B, uint32_t pt0,
                           int32_t* S, int* fault, uint8_t* sm, TcBars& bar, uint32_t tmem,
                           volatile int* abort, uint32_t pre) {
  constexpr uint32_t R = ring_of(N), kB = 2 * N * 128;  // ring slots, plane bytes of a stage
  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t m0 = blockIdx.x * kBM;
  const uint32_t kg0 = blockIdx.z * KG / gridDim.z, kg1 = (blockIdx.z + 1) * KG / gridDim.z;
  const uint32_t ns = kg1 - kg0, ngroups = (ns + kFlushGroups - 1) / kFlushGroups;
  uint8_t* au8 = sm;
  uint8_t* bsm = au8 + R * kAu8;
  if (warp == kTcConvWarps) {  // producer
    if (lane != 0) return;
    const uint32_t a_bytes = min(kBM, rows - m0) * kBK;
    for (uint32_t s = 0; s < ns; ++s) {
      const uint32_t slot = s % R, kg = kg0 + s;
      if (s >= R) mb_wait(&bar.empty[slot], ((s - R) / R) & 1u, abort);
      if (*abort) return;
      // the first `pre` stages' weight bytes were requested before the wait
      mb_expect_tx(&bar.full[slot], (s < pre ? 0u : a_bytes) + N * 256);
      if (s >= pre) bulk_copy(au8 + slot * kAu8, W + ((size_t)kg * rows + m0) * kBK, a_bytes, &bar.full[slot]);
      // plane tiles of 64 rows: atom column a of tile t -> rows 64 t .. of atom column a
#pragma unroll
      for (uint32_t t = 0; t < N / kBN; ++t)
#pragma unroll
        for (uint32_t a = 0; a < 2; ++a)
          bulk_copy(bsm + slot * kB + a * (N * 128) + t * (kBN * 128),
                    B + ((size_t)(pt0 + t) * KG + kg) * kBTile + a * (kBN * 128), kBN * 128,
                    &bar.full[slot]);
    }
    return;
  }
  if (warp == kTcConvWarps + 1) {  // MMA issuer
    if (lane != 0) return;
    for (uint32_t s = 0; s < ns; ++s) {
      const uint32_t slot = s % R, fb = s & 1u, g = s / kFlushGroups;
      mb_wait(&bar.full[slot], (s / R) & 1u, abort);
      mb_wait(&bar.conv[fb], (s >> 1) & 1u, abort);
      if (s % kFlushGroups == 0 && g >= 2) mb_wait(&bar.accfree[g & 1u], ((g - 2) >> 1) & 1u, abort);
      if (*abort) return;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t ta = tmem + (fb ? kAColB : kAColA), bbase = smem_addr(bsm + slot * kB);
      const uint32_t acc_tmem = tmem + (g & 1u) * kAccCols;
#pragma unroll
      for (uint32_t kk = 0; kk < 8; ++kk) {  // K 16 kk .. : eight columns of A, 32 bytes of B rows
        const uint64_t db = smem_desc(bbase + (kk >> 2) * (N * 128) + (kk & 3u) * 32);
        const uint32_t accumulate = (s % kFlushGroups != 0 || kk != 0) ? 1u : 0u;
        mma_f16_ts(acc_tmem, ta + 8 * kk, db, mma_idesc(N), accumulate);
      }
      mma_commit(&bar.empty[slot]);
      mma_commit(&bar.f16free[fb]);
      if ((s + 1) % kFlushGroups == 0 || s + 1 == ns) mma_commit(&bar.accf[g & 1u]);
    }
    return;
  }
  // converters
  int32_t iacc[N / 2];
#pragma unroll
  for (uint32_t i = 0; i < N / 2; ++i) iacc[i] = 0;
  uint32_t drained = 0;
  auto drain_group = [&](uint32_t gg) {
    mb_wait(&bar.accf[gg & 1u], (gg >> 1) & 1u, abort);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (!*abort) drain<N>(tmem + (gg & 1u) * kAccCols, iacc);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncwarp();
    if (lane == 0) mb_arrive(&bar.accfree[gg & 1u]);
  };
  for (uint32_t s = 0; s < ns; ++s) {
    const uint32_t slot = s % R, fb = s & 1u;
    mb_wait(&bar.full[slot], (s / R) & 1u, abort);
    if (s >= 2) mb_wait(&bar.f16free[fb], ((s - 2) >> 1) & 1u, abort);
    if (*abort) break;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    widen_to_tmem(au8 + slot * kAu8, tmem + (fb ? kAColB : kAColA));
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncwarp();
    if (lane == 0) mb_arrive(&bar.conv[fb]);
    // group g - 1 finished a stage ago: drain it while group g fills the other buffer
    const uint32_t g = s / kFlushGroups;
    if (s % kFlushGroups == 1 && g >= 1 && drained == g - 1) drain_group(drained++);
  }
  for (; drained < ngroups && !*abort; ++drained) drain_group(drained);
  if (*abort) {
    if (tid == 0) atomicExch(fault, 1);
    return;
  }
  // warp w holds rows 32 (w % 4) + lane, columns of half w / 4
  const uint32_t r = m0 + 32 * (warp & 3u) + lane;
  if (r >= rows) return;
  const uint32_t n0 = pt0 * kBN + (warp >> 2) * (N / 2);
#pragma unroll
  for (uint32_t i = 0; i < N / 2; ++i) {
    int32_t* dst = S + (size_t)(n0 + i) * rows + r;
    if (gridDim.z > 1)
      atomicAdd(dst, iacc[i]);
    else
      *dst = iacc[i];
  }
}

// One block: 128 rows of the matrix x up to kTN plane columns (blockIdx.y), tcgen05 MMAs.
// Before the dependency wait (nothing of it reads what the previous kernel writes): the
// barriers, the tensor memory, and, in the blocks of the first plane tile (the one the usual
// three planes fill), the weight bytes of the first three stages (model data).  A block that
// turns out to have no plane columns waits for those copies before it leaves.
__global__ void __launch_bounds__(kTcThreads, 1) k_bgemm(const uint8_t* gate, const uint8_t* W,
                                                         uint32_t rows, uint32_t KG, const uint8_t* B,
                                                         uint32_t Npad, const unsigned long long* orw,
                                                         int32_t* S, int* fault) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ TcBars bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const uint32_t tid = threadIdx.x, warp = tid >> 5;
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t nt = blockIdx.y;
  const uint32_t m0 = blockIdx.x * kBM;
  const uint32_t kg0 = blockIdx.z * KG / gridDim.z, kg1 = (blockIdx.z + 1) * KG / gridDim.z;
  const uint32_t pre = nt == 0 ? min(3u, kg1 - kg0) : 0u;  // stages whose weights go out early
  if (tid == 0) {
    for (uint32_t i = 0; i < kRing; ++i) {
      mb_init(&bar.full[i], 1);
      mb_init(&bar.empty[i], 1);
    }
    for (uint32_t i = 0; i < 2; ++i) {
      mb_init(&bar.conv[i], kTcConvWarps);
      mb_init(&bar.f16free[i], 1);
      mb_init(&bar.accf[i], 1);
      mb_init(&bar.accfree[i], kTcConvWarps);
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint32_t a_bytes = min(kBM, rows - m0) * kBK;
    for (uint32_t s = 0; s < pre; ++s) {
      mb_expect_only(&bar.full[s], a_bytes);
      bulk_copy(sm + s * kAu8, W + ((size_t)(kg0 + s) * rows + m0) * kBK, a_bytes, &bar.full[s]);
    }
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_addr(&tmem_slot)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_slot;
  pdl_enter();
  const int L = running(gate) ? limbs_of_or(*orw) : 0;
  const uint32_t cols = (uint32_t)L * Npad;  // plane columns in use (a multiple of 64)
  if (nt * kTN >= cols) {
    // nothing to compute: the early copies complete on their barriers' arrivals before the
    // block leaves (a wait that runs out leaves it all the same)
    if (tid == 0) {
      for (uint32_t s = 0; s < pre; ++s) {
        mb_arrive(&bar.full[s]);
        mb_wait(&bar.full[s], 0, &abort_flag);
      }
    }
  } else if (cols - nt * kTN <= kBN) {  // a last tile of 64 columns
    bgemm_tile<kBN>(W, rows, KG, B, nt * (kTN / kBN), S, fault, sm, bar, tmem, &abort_flag, pre);
  } else if (cols - nt * kTN <= 2 * kBN) {  // of 128
    bgemm_tile<2 * kBN>(W, rows, KG, B, nt * (kTN / kBN), S, fault, sm, bar, tmem, &abort_flag, pre);
  } else {
    bgemm_tile<kTN>(W, rows, KG, B, nt * (kTN / kBN), S, fault, sm, bar, tmem, &abort_flag, pre);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// ------------------------------------------------------------------ epilogues

struct BEpiParams {
  const uint8_t* gate;
  const RowDesc* rdesc;
  const int32_t* S;
  uint32_t rows, Npad, P;
  const unsigned long long* orw;  // the input vector's OR word (its plane count)
  const uint32_t* scale;
  int mode;
  // QKV (each row's keys and values go to its run's cache, at its position)
  int64_t* Q;                     // [P][dim] rotated queries
  const int32_t* rope;
  uint32_t dim, kv_dim, head_dim, layer;
  // residual: X[n][r] += y;  SiLU: H[n][j] = (silu(y_2j) * y_2j+1) >> 16
  int64_t* X;
  int64_t* H;
  uint32_t hidden;
  const int32_t* silu_tab;
  unsigned long long* or_out;     // SiLU, residual with norm: the output vector's OR word
  // residual followed by the next RMS normalization (k_bresnorm): its weights and output
  int64_t* XB;
  const int32_t* norm_w;
};

// y[n][r] = ((sum_k S_k[n][r] << 8k) * scale[r]) >> 24, wrapping, for rows r and r + 1 (r
// even; r + 1 only when it exists): every plane's pair of sums is requested before any is
// used, so the loads overlap instead of following one another.
__device__ __forceinline__ void combine_pair(const BEpiParams& p, int L, uint32_t n, uint32_t r, int64_t& y0,
                                             int64_t& y1) {
  const bool two = r + 1 < p.rows, paired = two && (p.rows & 1u) == 0;  // 8-byte aligned pairs
  int2 v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int32_t* src = p.S + ((size_t)k * p.Npad + n) * p.rows + r;
    v[k] = k >= L   ? make_int2(0, 0)
           : paired ? *reinterpret_cast<const int2*>(src)
                    : make_int2(src[0], two ? src[1] : 0);
  }
  const uint32_t s0 = __ldg(p.scale + r), s1 = two ? __ldg(p.scale + r + 1) : 0u;
  unsigned long long a0 = 0, a1 = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    a0 += (unsigned long long)(long long)v[k].x << (8 * k);
    a1 += (unsigned long long)(long long)v[k].y << (8 * k);
  }
  y0 = (int64_t)(a0 * (unsigned long long)s0) >> 24;
  y1 = (int64_t)(a1 * (unsigned long long)s1) >> 24;
}

// One thread per (position, row pair): rows 2i and 2i+1 are a rotary pair in Q and K and a
// gate/up pair in the feed-forward matrix.  Logits (an odd count possible) are written to
// the states of the rows that generate a token.
__global__ void __launch_bounds__(kRowThreads) k_bepi(const BEpiParams p) {
  __shared__ unsigned long long red[kRowThreads / 32];
  pdl_enter();
  if (!running(p.gate)) return;
  const int L = limbs_of_or(*p.orw);
  const uint32_t pairs = (p.rows + 1) / 2, items = p.P * pairs;  // below 2^32
  unsigned long long o = 0;
  for (uint32_t idx = blockIdx.x * blockDim.x + threadIdx.x; idx < items; idx += gridDim.x * blockDim.x) {
    const uint32_t n = idx / pairs, r = 2 * (idx - n * pairs);
    if (p.mode == kBEpiLogits) {
      const RowDesc rd = p.rdesc[n];
      if (!rd.generating) continue;
      int64_t* lg = reinterpret_cast<int64_t*>(rd.st + rd.off_logits);
      int64_t y0, y1;
      combine_pair(p, L, n, r, y0, y1);
      lg[r] = y0;
      if (r + 1 < p.rows) lg[r + 1] = y1;
      continue;
    }
    int64_t y0, y1;
    combine_pair(p, L, n, r, y0, y1);
    if (p.mode == kBEpiResid) {
      int64_t* x = p.X + (size_t)n * p.rows + r;
      x[0] = wadd(x[0], y0);
      x[1] = wadd(x[1], y1);
    } else if (p.mode == kBEpiSiLU) {
      const int64_t h = wmul(silu_lookup(y0, p.silu_tab), y1) >> 16;
      p.H[(size_t)n * p.hidden + (r >> 1)] = h;
      o |= (unsigned long long)(h ^ (h >> 63));
    } else {
      const RowDesc rd = p.rdesc[n];
      const uint32_t pos = rd.pos;
      uint8_t* st = rd.st;
      const int32_t* rope = p.rope + (size_t)pos * p.head_dim;  // [pos][head/2] pairs (cos, sin)
      if (r < p.dim) {
        const int32_t* cs = rope + ((r % p.head_dim) & ~1u);
        int64_t a2, b2;
        rotate_pair(y0, y1, __ldg(cs), __ldg(cs + 1), a2, b2);
        p.Q[(size_t)n * p.dim + r] = a2;
        p.Q[(size_t)n * p.dim + r + 1] = b2;
      } else if (r < p.dim + p.kv_dim) {
        const uint32_t e = r - p.dim;
        if (!fits_i32(y0)) record_error(st, err_key(pos, p.layer, 6, e));
        if (!fits_i32(y1)) record_error(st, err_key(pos, p.layer, 6, e + 1));
        const int32_t* cs = rope + ((e % p.head_dim) & ~1u);
        int64_t a2, b2;
        rotate_pair((int64_t)(int32_t)y0, (int64_t)(int32_t)y1, __ldg(cs), __ldg(cs + 1), a2, b2);
        if (!fits_i32(a2)) record_error(st, err_key(pos, p.layer, 8, e));
        if (!fits_i32(b2)) record_error(st, err_key(pos, p.layer, 8, e + 1));
        int32_t* kc = layer_cache(rd, rd.off_k, p.layer, p.kv_dim);
        kc[cache_word(e, pos, p.head_dim, rd.cache)] = (int32_t)a2;
        kc[cache_word(e + 1, pos, p.head_dim, rd.cache)] = (int32_t)b2;
      } else {
        const uint32_t e = r - p.dim - p.kv_dim;
        if (!fits_i32(y0)) record_error(st, err_key(pos, p.layer, 7, e));
        if (!fits_i32(y1)) record_error(st, err_key(pos, p.layer, 7, e + 1));
        int32_t* vc = layer_cache(rd, rd.off_v, p.layer, p.kv_dim);
        vc[cache_word(e, pos, p.head_dim, rd.cache)] = (int32_t)y0;
        vc[cache_word(e + 1, pos, p.head_dim, rd.cache)] = (int32_t)y1;
      }
    }
  }
  if (p.mode == kBEpiSiLU) block_or_to(o, p.or_out, red);
}

// Phases 11/16 and the normalization after them in one launch, one block per position row
// (kNormThreads threads): the residual X[n][r] += y[n][r] from the contraction's plane sums
// (as k_bepi's residual mode), then "RMS normalization" of the updated row into XB exactly as
// k_bnorm, the outputs' magnitudes ORed into *or_out.  Thread t takes the row pairs t,
// t + kNormThreads, ...; the first kNormPer / 2 of them stay in registers between the sum of
// squares and the division, the rest (rows beyond 4,096) are read back.
__global__ void __launch_bounds__(kNormThreads) k_bresnorm(const BEpiParams p) {
  __shared__ unsigned long long red[kNormThreads / 32];
  __shared__ InvDiv div;
  constexpr int kPairs = kNormPer / 2;
  const uint32_t d = p.rows, n = blockIdx.x;
  int32_t wv[kNormPer];
#pragma unroll
  for (int j = 0; j < kNormPer; ++j) {
    const uint32_t e = 2 * (threadIdx.x + (j >> 1) * kNormThreads) + (j & 1);
    wv[j] = e < d ? __ldg(p.norm_w + e) : 0;
  }
  const InvDiv Dd = make_invdiv_fast(d);  // floor(ss / d) by a multiply
  pdl_enter();
  if (!running(p.gate)) return;
  const int L = limbs_of_or(*p.orw);
  int64_t* x = p.X + (size_t)n * d;
  int64_t* y = p.XB + (size_t)n * d;
  int64_t xv[kNormPer];
  unsigned long long ss = 0;
#pragma unroll
  for (int j = 0; j < kPairs; ++j) {
    const uint32_t r = 2 * (threadIdx.x + j * kNormThreads);
    xv[2 * j] = xv[2 * j + 1] = 0;
    if (r < d) {
      int64_t y0, y1;
      combine_pair(p, L, n, r, y0, y1);
      xv[2 * j] = wadd(x[r], y0);
      x[r] = xv[2 * j];
      if (r + 1 < d) {
        xv[2 * j + 1] = wadd(x[r + 1], y1);
        x[r + 1] = xv[2 * j + 1];
      }
    }
    ss += (unsigned long long)xv[2 * j] * (unsigned long long)xv[2 * j] +
          (unsigned long long)xv[2 * j + 1] * (unsigned long long)xv[2 * j + 1];
  }
  for (uint32_t r = 2 * (threadIdx.x + kPairs * kNormThreads); r < d; r += 2 * kNormThreads) {
    int64_t y0, y1;
    combine_pair(p, L, n, r, y0, y1);
    const int64_t a = wadd(x[r], y0);
    x[r] = a;
    ss += (unsigned long long)a * (unsigned long long)a;
    if (r + 1 < d) {
      const int64_t b = wadd(x[r + 1], y1);
      x[r + 1] = b;
      ss += (unsigned long long)b * (unsigned long long)b;
    }
  }
  ss = block_sum(ss, red);  // (its barriers also order the residual stores before the reads below)
  if (threadIdx.x == 0) {
    uint64_t rms = isqrt_u64(udiv_inv(ss, Dd) + 42950ull);
    if (rms < 1) rms = 1;
    div = make_invdiv_fast((uint32_t)rms);
  }
  __syncthreads();
  const InvDiv D = div;
  unsigned long long o = 0;
#pragma unroll
  for (int j = 0; j < kNormPer; ++j) {
    const uint32_t e = 2 * (threadIdx.x + (j >> 1) * kNormThreads) + (j & 1);
    if (e < d) {
      const int64_t v = sdiv_trunc(wmul(xv[j], (int64_t)wv[j]), D) >> 8;
      y[e] = v;
      o |= (unsigned long long)(v ^ (v >> 63));
    }
  }
  for (uint32_t e = 2 * (threadIdx.x + kPairs * kNormThreads); e < d; e += 2 * kNormThreads)
    for (uint32_t u = 0; u < 2 && e + u < d; ++u) {
      const int64_t v = sdiv_trunc(wmul(x[e + u], (int64_t)__ldg(p.norm_w + e + u)), D) >> 8;
      y[e + u] = v;
      o |= (unsigned long long)(v ^ (v >> 63));
    }
  block_or_to(o, p.or_out, red);
}

// ------------------------------------------------------------------ attention

struct BAttnParams {
  const uint8_t* gate;
  const RowDesc* rdesc;
  const int64_t* Q;     // [P][dim]
  int64_t* O;           // [P][dim]
  const uint32_t* exp_tab;
  uint32_t layer, dim, heads, kv_heads, head_dim, kv_dim, inv_sqrt;
  unsigned long long* or_out;
};

constexpr int kAttnWarps = kRowThreads / 32;

constexpr int kAttnBatch = 8;  // positions a lane group loads at once

// Shared memory: the first round of value rows (each thread's kAttnBatch 16-byte chunks,
// copied when the kernel starts), then queries, per-warp partials, reduction slots and the
// row's scores.
constexpr size_t kAttnVpre = (size_t)kAttnBatch * kRowThreads * 16;
size_t battn_smem(uint32_t hd, uint32_t positions) {
  return kAttnVpre + 8 * ((size_t)hd * (1 + kAttnWarps) + kAttnWarps + positions);
}

__device__ __forceinline__ void battn_cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n\tcp.async.commit_group;" ::"r"(smem_addr(dst)),
               "l"(src)
               : "memory");
}

// Phase 9 for row blockIdx.y and head blockIdx.x ("Attention, stage by stage"), over its
// run's cache positions 0 .. pos: scores and their maximum, exponentials and their sum,
// probabilities with 24 fraction bits, and the weighted values with one >> 24.  Each lane
// group loads kAttnBatch positions a round; the first round's values are copied into shared
// memory together with its keys, so that they have arrived when the probabilities are known.
// The probabilities (e << 24) / Z come from a single-precision estimate of 1 / Z and exact
// corrections (e <= Z, Z below 2^46).  When every query element fits 32 signed bits,
// each product q * k is exact in one 32 x 32 -> 64-bit multiply-add (the same low 64 bits
// as the wrapping product), and so is every P * v (P <= 2^24).
__global__ void __launch_bounds__(kRowThreads) k_battn(const BAttnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_enter();
  if (!running(p.gate)) return;
  const uint32_t hd = p.head_dim, h = blockIdx.x, n = blockIdx.y;
  const RowDesc rd = p.rdesc[n];
  const uint32_t np = rd.pos + 1;
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int4* vpre = reinterpret_cast<int4*>(smem);                                  // [kAttnBatch][threads]
  int64_t* q_s = reinterpret_cast<int64_t*>(smem + kAttnVpre);
  unsigned long long* part = reinterpret_cast<unsigned long long*>(q_s + hd);  // [warps][hd]
  long long* red = reinterpret_cast<long long*>(part + (size_t)kAttnWarps * hd);
  long long* sc = red + kAttnWarps;                                            // [np]
  const uint32_t kvh = h / (p.heads / p.kv_heads);
  const int32_t* Kh = layer_cache(rd, rd.off_k, p.layer, p.kv_dim) + (size_t)kvh * rd.cache * hd;
  const int32_t* Vh = layer_cache(rd, rd.off_v, p.layer, p.kv_dim) + (size_t)kvh * rd.cache * hd;
  const uint32_t lpp = hd / 4, ppw = 32 / lpp;  // lanes per position (four elements each)
  const uint32_t sub = lane % lpp, slot = lane / lpp, e0 = sub * 4;
  const uint32_t round = kAttnWarps * ppw * kAttnBatch;
  // the first round: keys into registers, values into shared memory, before the queries
  int4 k4[kAttnBatch];
#pragma unroll
  for (int bb = 0; bb < kAttnBatch; ++bb) {
    const uint32_t tl = (bb * kAttnWarps + warp) * ppw + slot;
    k4[bb] = tl < np ? *reinterpret_cast<const int4*>(Kh + (size_t)tl * hd + e0) : make_int4(0, 0, 0, 0);
    if (tl < np) battn_cp16(vpre + bb * kRowThreads + tid, Vh + (size_t)tl * hd + e0);
  }
  int wide = 0;
  for (uint32_t i = tid; i < hd; i += kRowThreads) {
    const int64_t v = p.Q[(size_t)n * p.dim + (size_t)h * hd + i];
    q_s[i] = v;
    wide |= ((v ^ (v >> 63)) >> 31) != 0;
  }
  const bool q32 = !__syncthreads_or(wide);
  const int64_t q0 = q_s[e0], q1 = q_s[e0 + 1], q2 = q_s[e0 + 2], q3 = q_s[e0 + 3];
  const int32_t n0 = (int32_t)q0, n1 = (int32_t)q1, n2 = (int32_t)q2, n3 = (int32_t)q3;

  long long lmax = LLONG_MIN;
  for (uint32_t base = 0; base < np; base += round) {
    if (base != 0) {
#pragma unroll
      for (int bb = 0; bb < kAttnBatch; ++bb) {
        const uint32_t tl = base + (bb * kAttnWarps + warp) * ppw + slot;
        k4[bb] = tl < np ? *reinterpret_cast<const int4*>(Kh + (size_t)tl * hd + e0) : make_int4(0, 0, 0, 0);
      }
    }
    unsigned long long d[kAttnBatch];
#pragma unroll
    for (int bb = 0; bb < kAttnBatch; ++bb) {
      if (q32)
        d[bb] = (unsigned long long)((long long)n0 * k4[bb].x) + (unsigned long long)((long long)n1 * k4[bb].y) +
                (unsigned long long)((long long)n2 * k4[bb].z) + (unsigned long long)((long long)n3 * k4[bb].w);
      else
        d[bb] = (unsigned long long)q0 * (unsigned long long)(long long)k4[bb].x +
                (unsigned long long)q1 * (unsigned long long)(long long)k4[bb].y +
                (unsigned long long)q2 * (unsigned long long)(long long)k4[bb].z +
                (unsigned long long)q3 * (unsigned long long)(long long)k4[bb].w;
    }
    for (uint32_t o = lpp >> 1; o > 0; o >>= 1) {
#pragma unroll
      for (int bb = 0; bb < kAttnBatch; ++bb) d[bb] += __shfl_xor_sync(0xffffffffu, d[bb], o);
    }
#pragma unroll
    for (int bb = 0; bb < kAttnBatch; ++bb) {
      const uint32_t tl = base + (bb * kAttnWarps + warp) * ppw + slot;
      if (tl < np && sub == 0) {
        long long sv = (long long)d[bb] >> 16;
        sv = (long long)((unsigned long long)sv * (unsigned long long)p.inv_sqrt) >> 24;
        sc[tl] = sv;
        lmax = sv > lmax ? sv : lmax;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const long long v = __shfl_xor_sync(0xffffffffu, lmax, o);
    lmax = v > lmax ? v : lmax;
  }
  if (lane == 0) red[warp] = lmax;
  __syncthreads();
  long long m = red[0];
  for (int w = 1; w < kAttnWarps; ++w) m = red[w] > m ? red[w] : m;
  __syncthreads();

  unsigned long long z = 0;
  for (uint32_t tl = tid; tl < np; tl += kRowThreads) {
    unsigned long long idx = ((unsigned long long)m - (unsigned long long)sc[tl]) >> 8;
    if (idx > 4096) idx = 4096;
    const unsigned long long e = __ldg(p.exp_tab + idx);
    sc[tl] = (long long)e;
    z += e;
  }
  z = bwarp_sum(z);
  if (lane == 0) red[warp] = (long long)z;
  __syncthreads();
  unsigned long long Z = 0;
  for (int w = 0; w < kAttnWarps; ++w) Z += (unsigned long long)red[w];
  const float rz = rcp_estimate((float)Z);  // Z >= 2^30: the largest score's entry is 2^30
  for (uint32_t tl = tid; tl < np; tl += kRowThreads)
    sc[tl] = (long long)div_by_estimate((unsigned long long)sc[tl] << 24, Z, rz);
  __syncthreads();
  asm volatile("cp.async.wait_group 0;" ::: "memory");  // this thread's first-round values

  unsigned long long a0 = 0, a1 = 0, a2 = 0, a3 = 0;
  for (uint32_t base = 0; base < np; base += round) {
    int4 v4[kAttnBatch];
    int32_t pb[kAttnBatch];
#pragma unroll
    for (int bb = 0; bb < kAttnBatch; ++bb) {
      const uint32_t tl = base + (bb * kAttnWarps + warp) * ppw + slot;
      v4[bb] = tl >= np     ? make_int4(0, 0, 0, 0)
               : base == 0 ? vpre[bb * kRowThreads + tid]
                           : *reinterpret_cast<const int4*>(Vh + (size_t)tl * hd + e0);
      pb[bb] = tl < np ? (int32_t)sc[tl] : 0;  // P <= 2^24
    }
#pragma unroll
    for (int bb = 0; bb < kAttnBatch; ++bb) {
      a0 += (unsigned long long)((long long)pb[bb] * v4[bb].x);
      a1 += (unsigned long long)((long long)pb[bb] * v4[bb].y);
      a2 += (unsigned long long)((long long)pb[bb] * v4[bb].z);
      a3 += (unsigned long long)((long long)pb[bb] * v4[bb].w);
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
  __syncthreads();
  unsigned long long orv = 0;
  for (uint32_t j = tid; j < hd; j += kRowThreads) {
    unsigned long long s = 0;
    for (int w = 0; w < kAttnWarps; ++w) s += part[(size_t)w * hd + j];
    const long long v = (long long)s >> 24;
    p.O[(size_t)n * p.dim + (size_t)h * hd + j] = v;
    orv |= (unsigned long long)(v ^ (v >> 63));
  }
  block_or_to(orv, p.or_out, reinterpret_cast<unsigned long long*>(red));
}

// ------------------------------------------------------------------ end of a pass

// Rows pos0 .. pos0+P-1 of one run.
__global__ void k_rows_fill(RowDesc* rows, RowDesc tmpl, uint32_t pos0, uint32_t P) {
  const uint32_t n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= P) return;
  RowDesc r = tmpl;
  r.pos = pos0 + n;
  rows[n] = r;
}

// A chunk of one run: the first failing position (a cache store that did not fit, error 8,
// or a prompt id outside the vocabulary, error 3) fails the state there; otherwise the last
// position's residual becomes the state's x and the cursor moves past the chunk.
__global__ void __launch_bounds__(kRowThreads) k_bfinish(uint8_t* st, const int64_t* X, int64_t* x,
                                                         uint32_t d, uint32_t pos0, uint32_t P,
                                                         const int32_t* rstat, const int* fault) {
  __shared__ uint32_t first_bad;
  if (!running(st)) return;
  if (*fault) {  // a contraction's wait ran out: nothing of the chunk is trusted
    __syncthreads();
    if (threadIdx.x == 0) {
      hdr<uint32_t>(st, kHError) = CK_CUDA_ERROR;
      hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
    }
    return;
  }
  const uint64_t key = hdr_ld<uint64_t>(st, kHErrKey);
  const uint32_t key_pos = key == kNoError ? 0xFFFFFFFFu : (uint32_t)(key >> 44);
  if (threadIdx.x == 0) {
    first_bad = 0xFFFFFFFFu;
    for (uint32_t n = 0; n < P; ++n)
      if (rstat[n]) {
        first_bad = pos0 + n;
        break;
      }
  }
  __syncthreads();  // every thread has read the header before thread 0 writes it
  const uint32_t bad = first_bad;
  if (bad != 0xFFFFFFFFu && bad <= key_pos) {
    if (threadIdx.x == 0) {
      hdr<uint64_t>(st, kHErrKey) = kNoError;  // that position stopped before any store
      hdr<uint32_t>(st, kHError) = CK_INVALID_STATE;
      hdr<uint32_t>(st, kHPosition) = bad;
      hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
    }
    return;
  }
  if (key != kNoError) {
    if (threadIdx.x == 0) {
      hdr<uint32_t>(st, kHError) = CK_ARITHMETIC;
      hdr<uint32_t>(st, kHPosition) = key_pos;
      hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
    }
    return;
  }
  for (uint32_t i = threadIdx.x; i < d; i += blockDim.x) x[i] = X[(size_t)(P - 1) * d + i];
  if (threadIdx.x == 0) hdr<uint32_t>(st, kHPosition) = pos0 + P;
}

constexpr int kFinishThreads = 256;

// A batch of runs, one block per row: the end of its position.  A failed store or a token
// outside the vocabulary fails that run; otherwise the residual becomes its x, and where the
// position generates, phase 19 ("Sampling": the maximum pass, and above temperature zero
// the sum and draw passes) chooses the token.  Every run's turn counter advances.
__global__ void __launch_bounds__(kFinishThreads) k_mfinish(const RowDesc* rows, const int64_t* X,
                                                            uint32_t d, uint32_t vocab,
                                                            const uint32_t* exp_tab,
                                                            const int32_t* rstat, const int* fault) {
  __shared__ unsigned long long gsum[kSampleGroups];
  __shared__ long long wv[kFinishThreads / 32];
  __shared__ uint32_t wi[kFinishThreads / 32];
  __shared__ long long max_v;
  __shared__ uint32_t max_i;
  const uint32_t n = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const RowDesc rd = rows[n];
  uint8_t* st = rd.st;
  const uint64_t key = hdr_ld<uint64_t>(st, kHErrKey);
  const int32_t bad = *fault ? CK_CUDA_ERROR : rstat[n];  // a contraction that gave up fails all
  __syncthreads();  // header read by all before thread 0 writes it
  if (threadIdx.x == 0) hdr<uint64_t>(st, kHTurns) = hdr_ld<uint64_t>(st, kHTurns) + 1;
  if (bad || key != kNoError) {
    if (threadIdx.x == 0) {
      if (bad == CK_INVALID_STATE) hdr<uint64_t>(st, kHErrKey) = kNoError;  // stopped before any store
      hdr<uint32_t>(st, kHError) = bad ? (uint32_t)bad : CK_ARITHMETIC;
      hdr<uint32_t>(st, kHPhase) = CK_PHASE_FAILED;
    }
    return;
  }
  int64_t* x = reinterpret_cast<int64_t*>(st + rd.off_x);
  for (uint32_t i = threadIdx.x; i < d; i += blockDim.x) x[i] = X[(size_t)n * d + i];
  if (!rd.generating) {
    if (threadIdx.x == 0) hdr<uint32_t>(st, kHPosition) = rd.pos + 1;
    return;
  }
  // maximum pass: the first largest logit
  const long long* lg = reinterpret_cast<const long long*>(st + rd.off_logits);
  long long bv = LLONG_MIN;
  uint32_t bi = 0xFFFFFFFFu;
  for (uint32_t i = threadIdx.x; i < vocab; i += blockDim.x) {
    const long long v = __ldcg(lg + i);
    if (bi == 0xFFFFFFFFu || v > bv) {
      bv = v;
      bi = i;
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
  if (lane == 0) {
    wv[warp] = bv;
    wi[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kFinishThreads / 32; ++w)
      if (wi[w] != 0xFFFFFFFFu && (wv[w] > bv || (wv[w] == bv && wi[w] < bi))) {
        bv = wv[w];
        bi = wi[w];
      }
    max_v = bv;
    max_i = bi;
  }
  __syncthreads();
  bv = max_v;
  bi = max_i;
  const uint32_t temp = hdr_ld<uint32_t>(st, kHTemp);
  unsigned long long gen_state = hdr_ld<unsigned long long>(st, kHSeed), z = 0, draw = 0;
  if (temp != 0) {
    const SampleOut so = block_sample(lg, vocab, bv, temp, exp_tab, gen_state, gsum,
                                      kFinishThreads / 32, [] { __syncthreads(); });
    bi = so.token;
    gen_state = so.state;
    z = so.sum;
    draw = so.draw;
  }
  if (threadIdx.x == 0) {
    const uint32_t gen = hdr_ld<uint32_t>(st, kHGenerated);
    reinterpret_cast<uint32_t*>(st + rd.off_out)[gen] = bi;
    hdr<uint32_t>(st, kHGenerated) = gen + 1;
    hdr<uint32_t>(st, kHLastTok) = bi;
    hdr<long long>(st, kHMaxLogit) = bv;
    hdr<unsigned long long>(st, kHSeed) = gen_state;
    hdr<unsigned long long>(st, kHExpSum) = z;
    hdr<unsigned long long>(st, kHDraw) = draw;
    const bool stop = (hdr_ld<uint32_t>(st, kHFlags) & CK_FLAG_STOP_TOKENS) && (bi == 1 || bi == 2);
    if (gen + 1 == hdr_ld<uint32_t>(st, kHMaxTok) || stop) hdr<uint32_t>(st, kHPhase) = CK_PHASE_DONE;
    hdr<uint32_t>(st, kHPosition) = rd.pos + 1;
  }
}

__global__ void k_gather_headers(const uint8_t* const* states, uint32_t n, uint8_t* out) {
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n * (kHeaderBytes / 8);
       i += gridDim.x * blockDim.x) {
    const uint32_t s = i / (kHeaderBytes / 8), w = i % (kHeaderBytes / 8);
    reinterpret_cast<uint64_t*>(out)[i] = reinterpret_cast<const uint64_t*>(states[s])[w];
  }
}

uint32_t pad64(uint32_t n) { return (n + 63u) & ~63u; }

struct WorkLayout {
  uint64_t X, XB, Q, O, H, B, S, orw, rows, rstat, ptrs, hdrs, fault, size;
};

WorkLayout work_layout(const PrefillModel& m, uint32_t cap) {
  const uint64_t Np = pad64(cap);
  const uint64_t kg_max = std::max(m.pitch_d, m.pitch_h) / kBK;
  const uint64_t rows_max = std::max<uint64_t>({(uint64_t)m.cfg.dim + 2ull * m.kv_dim,
                                                2ull * m.cfg.hidden, (uint64_t)m.cfg.vocab});
  WorkLayout w;
  uint64_t off = 0;
  auto take = [&](uint64_t bytes) { uint64_t o = off; off = align256(off + bytes); return o; };
  w.X = take(8 * Np * m.cfg.dim);
  w.XB = take(8 * Np * m.cfg.dim);
  w.Q = take(8 * Np * m.cfg.dim);
  w.O = take(8 * Np * m.cfg.dim);
  w.H = take(8 * Np * m.cfg.hidden);
  w.B = take(8 * (Np / kBN) * kg_max * kBTile);     // up to 8 planes
  w.S = take(4 * 8 * Np * rows_max);
  w.orw = take(8ull * (4 * m.cfg.layers + 1));
  w.rows = take(sizeof(RowDesc) * Np);
  w.rstat = take(4 * Np);
  w.ptrs = take(8 * Np);
  w.hdrs = take((uint64_t)kHeaderBytes * Np);
  w.fault = take(4);
  w.size = off;
  return w;
}

// Launches one of the per-layer kernels with programmatic stream serialization allowed (the
// kernel begins with pdl_enter).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The layers for P rows (phases 3 to 16), then, with `classify`, the final norm and the
// classifier rows into the logits of the rows that generate.
cudaError_t enqueue_rows(const PrefillModel& m, const uint8_t* gate, const WorkLayout& w,
                         uint8_t* work, uint32_t P, uint32_t max_positions, bool classify,
                         cudaStream_t s) {
  const ck_config& c = m.cfg;
  const uint32_t Npad = pad64(P);
  const uint32_t KGd = m.pitch_d / kBK, KGh = m.pitch_h / kBK;
  int64_t* X = reinterpret_cast<int64_t*>(work + w.X);
  int64_t* XB = reinterpret_cast<int64_t*>(work + w.XB);
  int64_t* Q = reinterpret_cast<int64_t*>(work + w.Q);
  int64_t* O = reinterpret_cast<int64_t*>(work + w.O);
  int64_t* H = reinterpret_cast<int64_t*>(work + w.H);
  uint8_t* B = work + w.B;
  int32_t* S = reinterpret_cast<int32_t*>(work + w.S);
  unsigned long long* orw = reinterpret_cast<unsigned long long*>(work + w.orw);
  const RowDesc* rows = reinterpret_cast<const RowDesc*>(work + w.rows);
  int32_t* rstat = reinterpret_cast<int32_t*>(work + w.rstat);
  int* fault = reinterpret_cast<int*>(work + w.fault);
  cudaError_t e;
  if ((e = cudaMemsetAsync(orw, 0, 8ull * (4 * c.layers + 1), s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(rstat, 0, 4ull * P, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(fault, 0, 4, s)) != cudaSuccess) return e;

  // column-range split of a contraction: as many ranges as keep the blocks (one an SM, for
  // the usual three planes) within one wave, each range at least one group of four column
  // groups; a second wave of a few blocks would double the launch
  auto splits_for = [&](uint32_t nrows, uint32_t KG) {
    const uint32_t base = ((nrows + kBM - 1) / kBM) * ((3 * Npad + kTN - 1) / kTN);
    uint32_t z = (uint32_t)m.num_sms / base;
    return std::max(1u, std::min(z, KG / kFlushGroups));
  };
  // the planes of a vector, clearing the output of the contraction that follows when it splits
  auto planes = [&](const int64_t* vec, uint32_t ld, uint32_t cols, uint32_t KG,
                    const unsigned long long* ow, uint32_t next_rows, uint32_t next_KG) {
    const uint32_t clear = splits_for(next_rows, next_KG) > 1 ? next_rows : 0u;
    // a thread per 8 columns of a position; at least a thread per 4 words of the clearing
    // (sized for the usual three planes)
    const uint64_t work_items = std::max<uint64_t>((uint64_t)Npad * KG * 16, 3ull * Npad * clear / 4);
    const uint32_t blocks = (uint32_t)std::min<uint64_t>((work_items + kRowThreads - 1) / kRowThreads, 4096);
    launch_pdl(k_bplanes, dim3(blocks), dim3(kRowThreads), 0, s, gate, vec, ld, P, cols, Npad, KG, ow, B, S, clear);
  };
  auto gemm = [&](const uint8_t* Wm, uint32_t nrows, uint32_t KG, const unsigned long long* ow) {
    const dim3 grid((nrows + kBM - 1) / kBM, (8 * Npad + kTN - 1) / kTN, splits_for(nrows, KG));
    launch_pdl(k_bgemm, grid, dim3(kTcThreads), kTcSmem, s, gate, Wm, nrows, KG, (const uint8_t*)B, Npad, ow, S, fault);
  };
  // a residual epilogue together with the normalization that follows it (one block a row)
  auto resnorm = [&](BEpiParams p, const int32_t* norm_w, unsigned long long* or_out) {
    p.gate = gate;
    p.rdesc = rows;
    p.S = S;
    p.Npad = Npad;
    p.P = P;
    p.XB = XB;
    p.norm_w = norm_w;
    p.or_out = or_out;
    launch_pdl(k_bresnorm, dim3(P), dim3(kNormThreads), 0, s, p);
  };
  auto epi = [&](BEpiParams p) {
    p.gate = gate;
    p.rdesc = rows;
    p.S = S;
    p.Npad = Npad;
    p.P = P;
    const uint64_t items = (uint64_t)P * ((p.rows + 1) / 2);
    const uint32_t blocks = (uint32_t)std::min<uint64_t>((items + kRowThreads - 1) / kRowThreads, 8192);
    launch_pdl(k_bepi, dim3(blocks), dim3(kRowThreads), 0, s, p);
  };

  k_bembed<<<P, kRowThreads, 0, s>>>(gate, rows, X, c.dim, m.embed, m.embed_scale, c.vocab, rstat);
  for (uint32_t l = 0; l < c.layers; ++l) {
    const DevLayer& Wl = m.layers[l];
    unsigned long long* o4 = orw + 4 * l;
    // phases 4-8: attention norm (after layer 0 done by the previous layer's last launch),
    // Q/K/V rows, checked cache stores, rotary
    if (l == 0)
      launch_pdl(k_bnorm, dim3(P), dim3(kNormThreads), 0, s, gate, (const int64_t*)X, XB, Wl.attn_norm, c.dim, o4 + 0);
    planes(XB, c.dim, c.dim, KGd, o4 + 0, c.dim + 2 * m.kv_dim, KGd);
    gemm(Wl.wqkv, c.dim + 2 * m.kv_dim, KGd, o4 + 0);
    BEpiParams pq = {};
    pq.rows = c.dim + 2 * m.kv_dim;
    pq.orw = o4 + 0;
    pq.scale = Wl.sqkv;
    pq.mode = kBEpiQKV;
    pq.Q = Q;
    pq.rope = m.rope;
    pq.dim = c.dim;
    pq.kv_dim = m.kv_dim;
    pq.head_dim = m.head_dim;
    pq.layer = l;
    epi(pq);
    // phase 9
    BAttnParams pa = {};
    pa.gate = gate;
    pa.rdesc = rows;
    pa.Q = Q;
    pa.O = O;
    pa.exp_tab = m.exp_tab;
    pa.layer = l;
    pa.dim = c.dim;
    pa.heads = c.heads;
    pa.kv_heads = c.kv_heads;
    pa.head_dim = m.head_dim;
    pa.kv_dim = m.kv_dim;
    pa.inv_sqrt = m.inv_sqrt;
    pa.or_out = o4 + 1;
    launch_pdl(k_battn, dim3(c.heads, P), dim3(kRowThreads), battn_smem(m.head_dim, max_positions), s, pa);
    // phases 10-11: output rows and the residual
    planes(O, c.dim, c.dim, KGd, o4 + 1, c.dim, KGd);
    gemm(Wl.wo, c.dim, KGd, o4 + 1);
    BEpiParams po = {};
    po.rows = c.dim;
    po.orw = o4 + 1;
    po.scale = Wl.so;
    po.mode = kBEpiResid;
    po.X = X;
    // phases 12-14: feed-forward norm (in the residual's launch), gate and up rows, SiLU gating
    resnorm(po, Wl.ffn_norm, o4 + 2);
    planes(XB, c.dim, c.dim, KGd, o4 + 2, 2 * c.hidden, KGd);
    gemm(Wl.w13, 2 * c.hidden, KGd, o4 + 2);
    BEpiParams pg = {};
    pg.rows = 2 * c.hidden;
    pg.orw = o4 + 2;
    pg.scale = Wl.s13;
    pg.mode = kBEpiSiLU;
    pg.H = H;
    pg.hidden = c.hidden;
    pg.silu_tab = m.silu_tab;
    pg.or_out = o4 + 3;
    epi(pg);
    // phases 15-16: down rows and the residual
    planes(H, c.hidden, c.hidden, KGh, o4 + 3, c.dim, KGh);
    gemm(Wl.w2, c.dim, KGh, o4 + 3);
    BEpiParams pd = {};
    pd.rows = c.dim;
    pd.orw = o4 + 3;
    pd.scale = Wl.s2;
    pd.mode = kBEpiResid;
    pd.X = X;
    if (l + 1 < c.layers)  // with the next layer's attention norm
      resnorm(pd, m.layers[l + 1].attn_norm, orw + 4 * (l + 1));
    else if (classify)     // with the final norm
      resnorm(pd, m.final_norm, orw + 4 * c.layers);
    else
      epi(pd);
  }
  if (classify) {
    // phases 17-18: final norm and classifier rows (written only for generating rows)
    unsigned long long* of = orw + 4 * c.layers;  // the final norm ran with the last residual
    planes(XB, c.dim, c.dim, KGd, of, c.vocab, KGd);
    gemm(m.cls, c.vocab, KGd, of);
    BEpiParams pc = {};
    pc.rows = c.vocab;
    pc.orw = of;
    pc.scale = m.cls_scale;
    pc.mode = kBEpiLogits;
    epi(pc);
  }
  return cudaGetLastError();
}

// The attention kernel's dynamic shared memory may use what its static variables leave.
size_t battn_dynamic_max(size_t smem_optin) {
  cudaFuncAttributes a;
  if (cudaFuncGetAttributes(&a, k_battn) != cudaSuccess) return 0;
  return smem_optin > a.sharedSizeBytes ? smem_optin - a.sharedSizeBytes : 0;
}

}  // namespace

size_t prefill_work_bytes(const PrefillModel& m, uint32_t cap) { return work_layout(m, cap).size; }

bool prefill_supported(const PrefillModel& m, uint32_t cache, size_t smem_optin) {
  const uint32_t hd = m.head_dim;
  if (hd % 4 || hd > 128 || hd < 4 || (32 % (hd / 4)) != 0) return false;  // attention lane layout
  if (m.cfg.heads % m.cfg.kv_heads) return false;
  if (m.pitch_d > 65536 || m.pitch_h > 65536) return false;               // i32 plane sums
  if (battn_smem(hd, cache) > battn_dynamic_max(smem_optin)) return false;
  if ((size_t)kTcSmem > smem_optin) return false;
  return true;
}

cudaError_t configure_prefill(size_t smem_optin) {
  cudaError_t e = cudaFuncSetAttribute(k_bgemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_battn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)battn_dynamic_max(smem_optin));
}

cudaError_t enqueue_prefill(const PrefillModel& m, uint8_t* st, const StateLayout& lay, uint32_t pos0,
                            uint32_t P, uint8_t* work, uint32_t cap, cudaStream_t s) {
  if (P == 0 || P > cap) return cudaErrorInvalidValue;
  const WorkLayout w = work_layout(m, cap);
  RowDesc t = {};
  t.st = st;
  t.cache = lay.cache;
  t.np = 0xFFFFFFFFu;  // every row is a prompt position
  t.generating = 0;
  t.off_prompt = lay.prompt;
  t.off_out = lay.out;
  t.off_x = lay.x;
  t.off_logits = lay.logits;
  t.off_k = lay.k;
  t.off_v = lay.v;
  RowDesc* rows = reinterpret_cast<RowDesc*>(work + w.rows);
  k_rows_fill<<<(P + 255) / 256, 256, 0, s>>>(rows, t, pos0, P);
  cudaError_t e = enqueue_rows(m, st, w, work, P, pos0 + P, false, s);
  if (e != cudaSuccess) return e;
  k_bfinish<<<1, kRowThreads, 0, s>>>(st, reinterpret_cast<const int64_t*>(work + w.X),
                                      reinterpret_cast<int64_t*>(st + lay.x), m.cfg.dim, pos0, P,
                                      reinterpret_cast<const int32_t*>(work + w.rstat),
                                      reinterpret_cast<const int*>(work + w.fault));
  return cudaGetLastError();
}

cudaError_t batch_gather_headers(const PrefillModel& m, uint8_t* const* host_states, uint32_t n,
                                 uint8_t* work, uint32_t cap, uint8_t* host_out, cudaStream_t s) {
  if (n == 0 || n > cap) return cudaErrorInvalidValue;
  const WorkLayout w = work_layout(m, cap);
  cudaError_t e = cudaMemcpyAsync(work + w.ptrs, host_states, 8ull * n, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  k_gather_headers<<<(n * (kHeaderBytes / 8) + 255) / 256, 256, 0, s>>>(
      reinterpret_cast<const uint8_t* const*>(work + w.ptrs), n, work + w.hdrs);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaMemcpyAsync(host_out, work + w.hdrs, (size_t)kHeaderBytes * n, cudaMemcpyDeviceToHost, s)) !=
      cudaSuccess)
    return e;
  return cudaStreamSynchronize(s);
}

cudaError_t upload_batch_rows(const PrefillModel& m, const RowDesc* host_rows, uint32_t n, uint8_t* work,
                              uint32_t cap, cudaStream_t s) {
  if (n == 0 || n > cap) return cudaErrorInvalidValue;
  const WorkLayout w = work_layout(m, cap);
  return cudaMemcpyAsync(work + w.rows, host_rows, sizeof(RowDesc) * n, cudaMemcpyHostToDevice, s);
}

cudaError_t enqueue_batch_kernels(const PrefillModel& m, uint32_t n, uint32_t max_positions, uint8_t* work,
                                  uint32_t cap, cudaStream_t s) {
  if (n == 0 || n > cap) return cudaErrorInvalidValue;
  const WorkLayout w = work_layout(m, cap);
  cudaError_t e;
  if ((e = enqueue_rows(m, nullptr, w, work, n, max_positions, true, s)) != cudaSuccess) return e;
  k_mfinish<<<n, kFinishThreads, 0, s>>>(reinterpret_cast<const RowDesc*>(work + w.rows),
                                         reinterpret_cast<const int64_t*>(work + w.X), m.cfg.dim,
                                         m.cfg.vocab, m.exp_tab,
                                         reinterpret_cast<const int32_t*>(work + w.rstat),
                                         reinterpret_cast<const int*>(work + w.fault));
  return cudaGetLastError();
}

}  // namespace ck
