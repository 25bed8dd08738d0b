// The matrix-row kernel: y[r] = ((sum_c byte[r][c] * x[c] - 128 * sum_c x[c]) * scale[r]) >> 24
// with every product and sum wrapping in 64 bits ("The inference core", "A matrix row").
//
// GB300 design.  One CTA per SM streams whole rows with 16-byte non-allocating loads.
// Before the rows, every CTA packs the input vector into shared memory as byte planes:
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
constexpr int kR = 4;  // rows a warp accumulates at once

struct Scratch {
  unsigned long long red[kWarps];
  unsigned long long red2[kWarps];
  InvDiv div;
  unsigned long long S;
  unsigned long long orv;
};

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

// Packs the input vector (optionally residual-added and RMS-normalised) into byte planes.
// Returns the wrapping sum of the vector in *S and the limb count.
__device__ int prologue(const MatrowParams& p, uint32_t* planes32, Scratch* sc,
                        unsigned long long* S_out) {
  const uint32_t n = p.cols, words = p.pitch / 4;
  if (p.pro == kProNorm) {
    // "RMS normalization": rms = isqrt(sum(x*x) / n + 42,950), at least 1.
    unsigned long long ss = 0, dummy = 0;
    for (uint32_t i = threadIdx.x; i < n; i += kThreads) {
      const int64_t x = load_x(p, i);
      if (p.res_out && blockIdx.x == 0) p.res_out[i] = x;
      ss += (unsigned long long)x * (unsigned long long)x;
    }
    block_sum_or(ss, dummy, sc);
    if (threadIdx.x == 0) {
      uint64_t rms = isqrt_u64(ss / n + 42950ull);
      if (rms < 1) rms = 1;
      sc->div = make_invdiv((uint32_t)rms);
    }
    __syncthreads();
  }
  const InvDiv D = sc->div;
  unsigned long long S = 0, orv = 0;
  for (uint32_t g = threadIdx.x; g < words; g += kThreads) {
    int64_t v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t i = 4 * g + e;
      int64_t val = 0;
      if (i < n) {
        if (p.pro == kProNorm) {
          // y = ((x * w) / rms) >> 8, the division truncating toward zero
          const int64_t prod = wmul(load_x(p, i), (int64_t)p.norm_w[i]);
          val = sdiv_trunc(prod, D) >> 8;
        } else {
          val = p.in[i];
        }
      }
      v[e] = val;
      S += (unsigned long long)val;
      orv |= (unsigned long long)(val ^ (val >> 63));
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t w = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) w |= (uint32_t)(((uint64_t)v[e] >> (8 * k)) & 0xFF) << (8 * e);
      planes32[k * words + g] = w;
    }
  }
  block_sum_or(S, orv, sc);
  int L = 1;
  while (L < 8 && (orv >> (8 * L - 1)) != 0) ++L;
  *S_out = S;
  return L;
}

// Epilogue for the row handled by this lane (lanes 0..kR-1 of the warp, row r0 + lane).
__device__ __forceinline__ void epilogue(const MatrowParams& p, uint32_t row, int64_t y,
                                         uint32_t pos) {
  const int lane = threadIdx.x & 31;
  const int64_t partner = (int64_t)__shfl_xor_sync(0xffffffffu, (unsigned long long)y, 1);
  if (lane >= kR || row >= p.rows) return;
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

// Rows of W: row-major with the given pitch, or (kGrouped) the model's column-group layout,
// where the 16-byte chunk at column c of row r sits at grouped_offset(rows, r, c).
template <int L, bool kGrouped>
__device__ void rows_loop(const MatrowParams& p, const uint8_t* planes, unsigned long long S,
                          uint32_t pos) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t pitch = p.pitch;
  const uint32_t groups = (p.rows + kR - 1) / kR;
  const uint32_t nw = gridDim.x * kWarps;
  for (uint32_t g = blockIdx.x * kWarps + warp; g < groups; g += nw) {
    const uint32_t r0 = g * kR;
    const uint8_t* wrow[kR];
    uint32_t rsw[kR];  // grouped: the row's chunk rotation, (row & 7) << 4
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      const uint32_t row = min(r0 + r, p.rows - 1);
      wrow[r] = kGrouped ? p.W + (size_t)row * kGroupCols : p.W + (size_t)row * pitch;
      rsw[r] = (row & 7u) << 4;
    }
    const size_t gstride = (size_t)p.rows * kGroupCols;  // grouped: bytes between column groups
    uint32_t acc[kR][L];
#pragma unroll
    for (int r = 0; r < kR; ++r)
#pragma unroll
      for (int k = 0; k < L; ++k) acc[r][k] = 0;
    for (uint32_t c = lane * 16; c < pitch; c += 512) {
      uint4 w[kR];
      if (kGrouped) {
        const size_t gbase = (size_t)(c >> 7) * gstride;
        const uint32_t chunk = c & 0x70u;
#pragma unroll
        for (int r = 0; r < kR; ++r) w[r] = ld_stream16(wrow[r] + gbase + (chunk ^ rsw[r]));
      } else {
#pragma unroll
        for (int r = 0; r < kR; ++r) w[r] = ld_stream16(wrow[r] + c);
      }
#pragma unroll
      for (int k = 0; k < L; ++k) {
        const uint4 xk = *reinterpret_cast<const uint4*>(planes + (size_t)k * pitch + c);
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          if (k < L - 1) {
            uint32_t a = acc[r][k];
            a = __dp4a(w[r].x, xk.x, a);
            a = __dp4a(w[r].y, xk.y, a);
            a = __dp4a(w[r].z, xk.z, a);
            a = __dp4a(w[r].w, xk.w, a);
            acc[r][k] = a;
          } else {
            int a = (int)acc[r][k];
            a = dp4a_us(w[r].x, xk.x, a);
            a = dp4a_us(w[r].y, xk.y, a);
            a = dp4a_us(w[r].z, xk.z, a);
            a = dp4a_us(w[r].w, xk.w, a);
            acc[r][k] = (uint32_t)a;
          }
        }
      }
    }
    unsigned long long sums[kR];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      unsigned long long a = 0;
#pragma unroll
      for (int k = 0; k < L; ++k) {
        const unsigned long long t = (k < L - 1) ? (unsigned long long)acc[r][k]
                                                 : (unsigned long long)(long long)(int)acc[r][k];
        a += t << (8 * k);
      }
      sums[r] = warp_sum(a);
    }
    unsigned long long mine = sums[0];
#pragma unroll
    for (int r = 1; r < kR; ++r)
      if (lane == r) mine = sums[r];
    const uint32_t row = r0 + (uint32_t)lane;
    int64_t y = 0;
    if (lane < kR && row < p.rows) {
      const unsigned long long t = (mine - (S << 7)) * (unsigned long long)__ldg(p.scale + row);
      y = (int64_t)t >> 24;
    }
    epilogue(p, row, y, pos);
  }
}

__global__ void __launch_bounds__(kThreads, 1) k_matrow(const MatrowParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  if (p.state && hdr_ld<uint32_t>(p.state, kHPhase) != CK_PHASE_RUNNING) return;
  const uint32_t pos = p.state ? hdr_ld<uint32_t>(p.state, kHPosition) : 0u;
  uint8_t* planes = smem;
  Scratch* sc = reinterpret_cast<Scratch*>(smem + 8 * (size_t)p.pitch);
  unsigned long long S;
  const int L = prologue(p, reinterpret_cast<uint32_t*>(planes), sc, &S);
  if (p.grouped) {
    switch (L) {
      case 1: rows_loop<1, true>(p, planes, S, pos); break;
      case 2: rows_loop<2, true>(p, planes, S, pos); break;
      case 3: rows_loop<3, true>(p, planes, S, pos); break;
      case 4: rows_loop<4, true>(p, planes, S, pos); break;
      case 5: rows_loop<5, true>(p, planes, S, pos); break;
      case 6: rows_loop<6, true>(p, planes, S, pos); break;
      case 7: rows_loop<7, true>(p, planes, S, pos); break;
      default: rows_loop<8, true>(p, planes, S, pos); break;
    }
  } else {
    switch (L) {
      case 1: rows_loop<1, false>(p, planes, S, pos); break;
      case 2: rows_loop<2, false>(p, planes, S, pos); break;
      case 3: rows_loop<3, false>(p, planes, S, pos); break;
      case 4: rows_loop<4, false>(p, planes, S, pos); break;
      case 5: rows_loop<5, false>(p, planes, S, pos); break;
      case 6: rows_loop<6, false>(p, planes, S, pos); break;
      case 7: rows_loop<7, false>(p, planes, S, pos); break;
      default: rows_loop<8, false>(p, planes, S, pos); break;
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
  const uint32_t groups = (p.rows + kR - 1) / kR;
  uint32_t blocks = (groups + kWarps - 1) / kWarps;
  if (blocks > (uint32_t)num_sms) blocks = (uint32_t)num_sms;
  if (blocks < 1) blocks = 1;
  k_matrow<<<blocks, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ck
