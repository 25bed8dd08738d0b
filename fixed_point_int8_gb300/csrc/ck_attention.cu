// Phase 9, attention for one query position ("The inference core", "Attention, stage by
// stage"), all heads at once.
//
// GB300 design.  One thread-block cluster per head; the cluster's CTAs split the p
// positions into contiguous chunks.  The four stages stay separate because the
// exponential is a table lookup of (largest score - score) >> 8, which cannot be rescaled
// online: each CTA computes its chunk's scores into shared memory, the cluster exchanges
// the chunk maxima through distributed shared memory, each CTA turns its scores into
// exponentials and a partial sum, the cluster exchanges the sums, each CTA forms its
// probabilities and the partial weighted sum of values, and rank 0 adds the partials and
// applies the single >> 24.  All sums are integer, so the split changes no bit.
//
// Two kernels share this plan.  For short caches a lane takes four elements of a cache row
// and keeps few registers, so CTAs fit beside the tail of the previous kernel; for long
// caches (more than 128 positions a CTA) a lane takes sixteen elements, keeps several rows'
// loads in flight and forms the wrapping products from 32-bit halves, cutting the
// instructions per position.
#include <climits>
#include <cooperative_groups.h>

#include "ck_internal.cuh"

namespace cg = cooperative_groups;

namespace ck {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kLongChunk = 128;  // positions a CTA may cover from which the long kernel runs

// A 16-byte cache load that bypasses L1: each cache word is read once per position.
__device__ __forceinline__ int4 ld_nc_int4(const int32_t* p) {
  int4 v;
  asm("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ long long warp_max(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const long long t = __shfl_xor_sync(0xffffffffu, v, o);
    v = t > v ? t : v;
  }
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Short caches: lanes per position = hd / 4, one cache load a lane per warp step.  Few
// registers, so that many CTAs fit an SM beside the tail of the previous kernel.
__global__ void __launch_bounds__(kThreads) k_attention_short(const AttnParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  // launched with programmatic dependent launch: wait for the kernels before this one on the
  // stream (the queries and the cache words they wrote), then let the next kernel start early
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (hdr_ld<uint32_t>(p.state, kHPhase) != CK_PHASE_RUNNING) return;  // whole cluster alike
  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t hd = p.head_dim;
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int64_t* q_s = reinterpret_cast<int64_t*>(smem);
  unsigned long long* part = reinterpret_cast<unsigned long long*>(q_s + hd);  // [kWarps][hd]
  unsigned long long* cpart = part + kWarps * hd;                               // [hd]
  long long* cmax = reinterpret_cast<long long*>(cpart + hd);                   // [1]
  unsigned long long* csum = reinterpret_cast<unsigned long long*>(cmax + 1);   // [1]
  long long* red = reinterpret_cast<long long*>(csum + 1);                      // [kWarps]
  long long* sc = red + kWarps;                                                 // [chunk_cap]

  const uint32_t pos = hdr_ld<uint32_t>(p.state, kHPosition);
  const uint32_t P = pos + 1;  // positions so far, the current one included
  const uint32_t h = blockIdx.x;
  const uint32_t rank = cluster.block_rank(), CL = cluster.num_blocks();
  const uint32_t kvh = h / (p.heads / p.kv_heads);  // "head h reads key/value head h/(heads/kvHeads)"
  const uint32_t cs = (P + CL - 1) / CL;
  const uint32_t t0 = min(P, rank * cs), t1 = min(P, t0 + cs);
  const uint32_t n = t1 - t0;

  for (uint32_t i = tid; i < hd; i += kThreads) q_s[i] = p.q[(size_t)h * hd + i];
  __syncthreads();

  const int32_t* Kh = p.kcache + (size_t)kvh * p.cache * hd;  // the head's positions, contiguous
  const int32_t* Vh = p.vcache + (size_t)kvh * p.cache * hd;
  const uint32_t lpp = hd / 4;       // lanes per position, four elements each
  const uint32_t ppw = 32 / lpp;     // positions per warp step
  const uint32_t sub = lane % lpp, slot = lane / lpp, e0 = sub * 4;
  const int64_t q0 = q_s[e0], q1 = q_s[e0 + 1], q2 = q_s[e0 + 2], q3 = q_s[e0 + 3];

  // stage 0: s_t = (((q . k_t) >> 16) * inv) >> 24, products and sums wrapping; keep the max
  long long lmax = LLONG_MIN;
  for (uint32_t base = warp * ppw; base < n; base += kWarps * ppw) {
    const uint32_t tl = base + slot;
    unsigned long long d = 0;
    if (tl < n) {
      const int4 k4 = *reinterpret_cast<const int4*>(Kh + (size_t)(t0 + tl) * hd + e0);
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
  lmax = warp_max(lmax);
  if (lane == 0) red[warp] = lmax;
  __syncthreads();
  if (tid == 0) {
    long long m = red[0];
    for (int w = 1; w < kWarps; ++w) m = red[w] > m ? red[w] : m;
    *cmax = m;
  }
  cluster.sync();
  long long m = LLONG_MIN;
  for (uint32_t r = 0; r < CL; ++r) {
    const long long v = *cluster.map_shared_rank(cmax, r);
    m = v > m ? v : m;
  }

  // stage 1: e_t = EXP[min((m - s_t) >> 8, 4096)]; the exact difference is >= 0 and fits u64
  unsigned long long z = 0;
  for (uint32_t tl = tid; tl < n; tl += kThreads) {
    unsigned long long idx = ((unsigned long long)m - (unsigned long long)sc[tl]) >> 8;
    if (idx > 4096) idx = 4096;
    const unsigned long long e = __ldg(p.exp_tab + idx);
    sc[tl] = (long long)e;
    z += e;
  }
  z = warp_sum(z);
  if (lane == 0) red[warp] = (long long)z;
  __syncthreads();
  if (tid == 0) {
    unsigned long long t = 0;
    for (int w = 0; w < kWarps; ++w) t += (unsigned long long)red[w];
    *csum = t;
  }
  cluster.sync();
  unsigned long long Z = 0;
  for (uint32_t r = 0; r < CL; ++r) Z += *cluster.map_shared_rank(csum, r);

  // stage 2: P_t = (e_t << 24) / Z, 24 fractional bits
  for (uint32_t tl = tid; tl < n; tl += kThreads)
    sc[tl] = (long long)(((unsigned long long)sc[tl] << 24) / Z);
  __syncthreads();

  // stage 3: sum over positions of P_t * v_t[j] (exact: |sum| < 2^55), then one >> 24
  unsigned long long a0 = 0, a1 = 0, a2 = 0, a3 = 0;
  for (uint32_t base = warp * ppw; base < n; base += kWarps * ppw) {
    const uint32_t tl = base + slot;
    if (tl < n) {
      const int4 v4 = *reinterpret_cast<const int4*>(Vh + (size_t)(t0 + tl) * hd + e0);
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
  __syncthreads();
  for (uint32_t j = tid; j < hd; j += kThreads) {
    unsigned long long s = 0;
    for (int w = 0; w < kWarps; ++w) s += part[(size_t)w * hd + j];
    cpart[j] = s;
  }
  cluster.sync();
  if (rank == 0) {
    for (uint32_t j = tid; j < hd; j += kThreads) {
      unsigned long long s = 0;
      for (uint32_t r = 0; r < CL; ++r) s += cluster.map_shared_rank(cpart, r)[j];
      p.o[(size_t)h * hd + j] = (long long)s >> 24;
    }
  }
  cluster.sync();  // peers keep their shared memory until rank 0 has read it
}

// Long caches: one cache row of hd = E * G elements is read by G lanes, E elements each: load i of lane
// `sub` covers elements i * 4G + 4 sub .. + 3, so the G lanes of a load read 16 G contiguous
// bytes.  A warp step covers 32 / G positions; kU steps' loads are in flight together.
template <int E>
__global__ void __launch_bounds__(kThreads) k_attention_long(const AttnParams p) {
  constexpr int kLoads = E / 4;     // 16-byte loads a lane makes per position
  constexpr int kU = 32 / E;        // warp steps whose loads are in flight together
  extern __shared__ __align__(16) uint8_t smem[];
  // launched with programmatic dependent launch: wait for the kernels before this one on the
  // stream (the queries and the cache words they wrote), then let the next kernel start early
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (hdr_ld<uint32_t>(p.state, kHPhase) != CK_PHASE_RUNNING) return;  // whole cluster alike
  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t hd = p.head_dim;
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int64_t* q_s = reinterpret_cast<int64_t*>(smem);
  unsigned long long* part = reinterpret_cast<unsigned long long*>(q_s + hd);  // [kWarps][hd]
  unsigned long long* cpart = part + kWarps * hd;                               // [hd]
  long long* cmax = reinterpret_cast<long long*>(cpart + hd);                   // [1]
  unsigned long long* csum = reinterpret_cast<unsigned long long*>(cmax + 1);   // [1]
  long long* red = reinterpret_cast<long long*>(csum + 1);                      // [kWarps]
  long long* sc = red + kWarps;                                                 // [chunk_cap]

  const uint32_t pos = hdr_ld<uint32_t>(p.state, kHPosition);
  const uint32_t P = pos + 1;  // positions so far, the current one included
  const uint32_t h = blockIdx.x;
  const uint32_t rank = cluster.block_rank(), CL = cluster.num_blocks();
  const uint32_t kvh = h / (p.heads / p.kv_heads);  // "head h reads key/value head h/(heads/kvHeads)"
  const uint32_t cs = (P + CL - 1) / CL;
  const uint32_t t0 = min(P, rank * cs), t1 = min(P, t0 + cs);
  const uint32_t n = t1 - t0;

  for (uint32_t i = tid; i < hd; i += kThreads) q_s[i] = p.q[(size_t)h * hd + i];
  __syncthreads();

  const int32_t* Kh = p.kcache + (size_t)kvh * p.cache * hd;  // the head's positions, contiguous
  const int32_t* Vh = p.vcache + (size_t)kvh * p.cache * hd;
  const uint32_t G = hd / E;          // lanes per position
  const uint32_t ppw = 32 / G;        // positions per warp step
  const uint32_t step = kWarps * ppw; // positions the CTA covers per warp step
  const uint32_t sub = lane % G, slot = lane / G;
  // this lane's query elements, split into 32-bit halves for the wrapping products
  uint32_t ql[E], qh[E];
#pragma unroll
  for (int i = 0; i < kLoads; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint64_t v = (uint64_t)q_s[i * 4 * G + 4 * sub + c];
      ql[4 * i + c] = (uint32_t)v;
      qh[4 * i + c] = (uint32_t)(v >> 32);
    }

  // stage 0: s_t = (((q . k_t) >> 16) * inv) >> 24, products and sums wrapping; keep the max.
  // q k mod 2^64 for a signed 32-bit k: the wide product of the low halves, plus
  // (q_hi k + q_lo (k >> 31)) in the upper 32 bits.
  long long lmax = LLONG_MIN;
  for (uint32_t base = warp * ppw; base < n; base += kU * step) {
    int4 kk[kU][kLoads];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const uint32_t tl = base + u * step + slot;
#pragma unroll
      for (int i = 0; i < kLoads; ++i)
        kk[u][i] = tl < n ? ld_nc_int4(Kh + (size_t)(t0 + tl) * hd + i * 4 * G + 4 * sub)
                          : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const uint32_t tl = base + u * step + slot;
      uint64_t lo = 0;
      uint32_t hi = 0;
#pragma unroll
      for (int i = 0; i < kLoads; ++i) {
        const int32_t kv[4] = {kk[u][i].x, kk[u][i].y, kk[u][i].z, kk[u][i].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t k = (uint32_t)kv[c];
          lo += (uint64_t)ql[4 * i + c] * k;
          hi += qh[4 * i + c] * k + ql[4 * i + c] * (uint32_t)(kv[c] >> 31);
        }
      }
      unsigned long long d = lo + ((uint64_t)hi << 32);
      for (uint32_t o = G >> 1; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      if (tl < n && sub == 0) {
        long long s = (long long)d >> 16;
        s = (long long)((unsigned long long)s * (unsigned long long)p.inv_sqrt) >> 24;
        sc[tl] = s;
        lmax = s > lmax ? s : lmax;
      }
    }
  }
  lmax = warp_max(lmax);
  if (lane == 0) red[warp] = lmax;
  __syncthreads();
  if (tid == 0) {
    long long m = red[0];
    for (int w = 1; w < kWarps; ++w) m = red[w] > m ? red[w] : m;
    *cmax = m;
  }
  cluster.sync();
  long long m = LLONG_MIN;
  for (uint32_t r = 0; r < CL; ++r) {
    const long long v = *cluster.map_shared_rank(cmax, r);
    m = v > m ? v : m;
  }

  // stage 1: e_t = EXP[min((m - s_t) >> 8, 4096)]; the exact difference is >= 0 and fits u64
  unsigned long long z = 0;
  for (uint32_t tl = tid; tl < n; tl += kThreads) {
    unsigned long long idx = ((unsigned long long)m - (unsigned long long)sc[tl]) >> 8;
    if (idx > 4096) idx = 4096;
    const unsigned long long e = __ldg(p.exp_tab + idx);
    sc[tl] = (long long)e;
    z += e;
  }
  z = warp_sum(z);
  if (lane == 0) red[warp] = (long long)z;
  __syncthreads();
  if (tid == 0) {
    unsigned long long t = 0;
    for (int w = 0; w < kWarps; ++w) t += (unsigned long long)red[w];
    *csum = t;
  }
  cluster.sync();
  unsigned long long Z = 0;
  for (uint32_t r = 0; r < CL; ++r) Z += *cluster.map_shared_rank(csum, r);

  // stage 2: P_t = (e_t << 24) / Z, 24 fractional bits; P_t <= 2^24 since e_t <= Z
  for (uint32_t tl = tid; tl < n; tl += kThreads)
    sc[tl] = (long long)(((unsigned long long)sc[tl] << 24) / Z);
  __syncthreads();

  // stage 3: sum over positions of P_t * v_t[j] (exact: |sum| < 2^55), then one >> 24.  P_t
  // fits 32 signed bits, so each product is one widening multiply.
  long long acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0;
  for (uint32_t base = warp * ppw; base < n; base += kU * step) {
    int4 vv[kU][kLoads];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const uint32_t tl = base + u * step + slot;
#pragma unroll
      for (int i = 0; i < kLoads; ++i)
        vv[u][i] = tl < n ? ld_nc_int4(Vh + (size_t)(t0 + tl) * hd + i * 4 * G + 4 * sub)
                          : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const uint32_t tl = base + u * step + slot;
      const int32_t pr = tl < n ? (int32_t)sc[tl] : 0;
#pragma unroll
      for (int i = 0; i < kLoads; ++i) {
        acc[4 * i + 0] += (long long)pr * vv[u][i].x;
        acc[4 * i + 1] += (long long)pr * vv[u][i].y;
        acc[4 * i + 2] += (long long)pr * vv[u][i].z;
        acc[4 * i + 3] += (long long)pr * vv[u][i].w;
      }
    }
  }
  // the lanes of one sub (one element set) add over the warp's slots
#pragma unroll
  for (int e = 0; e < E; ++e)
    for (uint32_t o = 16; o >= G; o >>= 1)
      acc[e] += (long long)__shfl_xor_sync(0xffffffffu, (unsigned long long)acc[e], o);
  if (slot == 0) {
#pragma unroll
    for (int i = 0; i < kLoads; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        part[(size_t)warp * hd + i * 4 * G + 4 * sub + c] = (unsigned long long)acc[4 * i + c];
  }
  __syncthreads();
  for (uint32_t j = tid; j < hd; j += kThreads) {
    unsigned long long s = 0;
    for (int w = 0; w < kWarps; ++w) s += part[(size_t)w * hd + j];
    cpart[j] = s;
  }
  cluster.sync();
  if (rank == 0) {
    for (uint32_t j = tid; j < hd; j += kThreads) {
      unsigned long long s = 0;
      for (uint32_t r = 0; r < CL; ++r) s += cluster.map_shared_rank(cpart, r)[j];
      p.o[(size_t)h * hd + j] = (long long)s >> 24;
    }
  }
  cluster.sync();  // peers keep their shared memory until rank 0 has read it
}

size_t attn_smem(uint32_t hd, uint32_t chunk_cap) {
  return 8 * ((size_t)hd * (2 + kWarps) + 2 + kWarps + chunk_cap);
}

}  // namespace

cudaError_t configure_attention() {
  const int kMax = 96 * 1024;
  cudaError_t e = cudaFuncSetAttribute(k_attention_short, cudaFuncAttributeMaxDynamicSharedMemorySize, kMax);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_attention_long<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMax);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_attention_long<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMax);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_attention_long<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMax);
  return e;
}

cudaError_t launch_attention(const AttnParams& p, cudaStream_t s, int cluster) {
  const size_t smem = attn_smem(p.head_dim, p.chunk_cap);
  if (smem > 96 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.heads, (unsigned)cluster, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)cluster;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // the kernel follows the state's capacity: a graph captured for the state serves every
  // position, and a CTA's share of the positions is at most chunk_cap
  if (p.chunk_cap < kLongChunk) return cudaLaunchKernelEx(&cfg, k_attention_short, p);
  if (p.head_dim >= 16) return cudaLaunchKernelEx(&cfg, k_attention_long<16>, p);
  if (p.head_dim == 8) return cudaLaunchKernelEx(&cfg, k_attention_long<8>, p);
  return cudaLaunchKernelEx(&cfg, k_attention_long<4>, p);
}

}  // namespace ck
