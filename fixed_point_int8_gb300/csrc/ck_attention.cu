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
#include <climits>
#include <cooperative_groups.h>

#include "ck_internal.cuh"

namespace cg = cooperative_groups;

namespace ck {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;  // warp steps whose cache loads are in flight together

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

// Shared memory: queries, per-warp and per-CTA partials, the cluster's chunk maxima and sums
// (slot r written by rank r), the two barriers those writes complete on, reduction slots, the
// chunk's scores, then (16-byte aligned) the first batch of value rows.
__host__ __device__ inline size_t attn_vpre_offset(uint32_t hd, uint32_t chunk_cap) {
  return (8 * ((size_t)hd * (2 + kWarps) + 18 + kWarps + chunk_cap) + 15) & ~(size_t)15;
}

// 16-byte asynchronous copy from global to shared memory (zeros and no read when not valid),
// and the wait for all of this thread's copies.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n\tcp.async.commit_group;" ::"r"(d), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Shared-memory barriers (mbarrier) and bulk copies into shared memory that complete on them.
__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void lbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void lbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void lbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
__device__ __forceinline__ bool lbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void lbulk(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(saddr(dst)),
      "l"(src), "r"(bytes), "r"(saddr(bar))
      : "memory");
}

// An eight-byte store into the same shared-memory variable of cluster peer `peer`, completing
// on that peer's barrier `bar` (the receiving CTA counts the bytes).
__device__ __forceinline__ void st_async_peer(void* local, unsigned long long v, uint64_t* bar, uint32_t peer) {
  uint32_t ra, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(saddr(local)), "r"(peer));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(saddr(bar)), "r"(peer));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(ra), "l"(v),
               "r"(rb)
               : "memory");
}
// Waits for an exchange's barrier (phase 0); a wait that runs out fails the state with error 9
// and the kernel goes on, so that every thread reaches the same barriers.
constexpr uint32_t kXPoll = 1u << 22;
__device__ __forceinline__ void exchange_wait(uint64_t* bar, uint8_t* state) {
  uint32_t i = 0;
  while (!lbar_try(bar, 0) && ++i < kXPoll) {
  }
  if (i >= kXPoll) {
    hdr<uint32_t>(state, kHError) = CK_CUDA_ERROR;
    hdr<uint32_t>(state, kHPhase) = CK_PHASE_FAILED;
  }
}

// Lanes per position = hd / 4, four elements a lane; a warp issues kUnroll steps' cache loads
// before it uses them.  The first batch of key rows of earlier positions is loaded into
// registers before the dependency wait, the first batch of value rows into shared memory
// (each lane copies what it reads back itself), the newest rows together with the queries
// after it.  64 registers a thread, so that four CTAs fit an SM: a head's cluster of eight
// is placed as soon as two SMs are free of the previous kernel.
__global__ void __launch_bounds__(kThreads, 4) k_attention(const AttnParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t hd = p.head_dim;
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int64_t* q_s = reinterpret_cast<int64_t*>(smem);
  unsigned long long* part = reinterpret_cast<unsigned long long*>(q_s + hd);  // [kWarps][hd]
  unsigned long long* cpart = part + kWarps * hd;                               // [hd]
  long long* cmax = reinterpret_cast<long long*>(cpart + hd);                   // [8]
  unsigned long long* csum = reinterpret_cast<unsigned long long*>(cmax + 8);   // [8]
  uint64_t* xbar = reinterpret_cast<uint64_t*>(csum + 8);                        // [2]
  long long* red = reinterpret_cast<long long*>(xbar + 2);                      // [kWarps]
  long long* sc = red + kWarps;                                                 // [chunk_cap]
  int4* vpre = reinterpret_cast<int4*>(smem + attn_vpre_offset(hd, p.chunk_cap));  // [kUnroll][kThreads]
  // The maxima and sums reach the peers as asynchronous remote stores that complete on the
  // receiving CTA's barrier (eight bytes from each CTA of the cluster).  Every CTA has set up
  // its barriers before any peer writes into it: the arrival here, the wait just before the
  // first such write.
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      lbar_init(&xbar[i], 1);
      lbar_expect_tx(&xbar[i], 8 * cluster.num_blocks());
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");

  // Launched with programmatic dependent launch.  Before the wait this kernel reads only what
  // was written before the previous kernel started: the position (set by the previous
  // position's last kernel) and the cache rows of earlier positions.  The queries and the
  // newest cache rows come from the kernel just before: after the wait.
  const uint32_t pos = hdr_ld<uint32_t>(p.state, kHPosition);
  const uint32_t P = pos + 1;  // positions so far, the current one included
  const uint32_t older = min(pos, p.cache);  // rows below this were written at earlier positions
  const uint32_t h = blockIdx.x;
  const uint32_t rank = cluster.block_rank(), CL = cluster.num_blocks();
  const uint32_t kvh = h / (p.heads / p.kv_heads);  // "head h reads key/value head h/(heads/kvHeads)"
  const uint32_t cs = (P + CL - 1) / CL;
  const uint32_t t0 = min(P, rank * cs), t1 = min(P, t0 + cs);
  const uint32_t n = t1 - t0;
  const int32_t* Kh = p.kcache + (size_t)kvh * p.cache * hd;  // the head's positions, contiguous
  const int32_t* Vh = p.vcache + (size_t)kvh * p.cache * hd;
  const uint32_t lpp = hd / 4;       // lanes per position, four elements each
  const uint32_t ppw = 32 / lpp;     // positions per warp step
  const uint32_t sub = lane % lpp, slot = lane / lpp, e0 = sub * 4;
  const uint32_t base0 = warp * ppw;
  int4 k4[kUnroll];  // the warp's first batch of keys (its values wait in vpre)
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const uint32_t tl = base0 + u * kWarps * ppw + slot;
    const bool early = tl < n && t0 + tl < older;
    k4[u] = early ? *reinterpret_cast<const int4*>(Kh + (size_t)(t0 + tl) * hd + e0) : make_int4(0, 0, 0, 0);
    if (early) cp_async16(vpre + u * kThreads + tid, Vh + (size_t)(t0 + tl) * hd + e0, true);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the newest rows of the first batch and the queries, requested together; the phase is
  // tested after them (the whole cluster reads the same header word and returns alike)
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const uint32_t tl = base0 + u * kWarps * ppw + slot;
    if (tl < n && t0 + tl >= older) {
      k4[u] = *reinterpret_cast<const int4*>(Kh + (size_t)(t0 + tl) * hd + e0);
      cp_async16(vpre + u * kThreads + tid, Vh + (size_t)(t0 + tl) * hd + e0, true);
    }
  }
  const bool running = hdr_ld<uint32_t>(p.state, kHPhase) == CK_PHASE_RUNNING;
  for (uint32_t i = tid; i < hd; i += kThreads) q_s[i] = p.q[(size_t)h * hd + i];
  if (!running) {
    cp_async_wait_all();  // no copy into shared memory outlives the CTA
    return;
  }
  __syncthreads();

  const int64_t q0 = q_s[e0], q1 = q_s[e0 + 1], q2 = q_s[e0 + 2], q3 = q_s[e0 + 3];

  // stage 0: s_t = (((q . k_t) >> 16) * inv) >> 24, products and sums wrapping; keep the max
  long long lmax = LLONG_MIN;
  for (uint32_t base = base0; base < n; base += kUnroll * kWarps * ppw) {
    if (base != base0) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t tl = base + u * kWarps * ppw + slot;
        k4[u] = tl < n ? *reinterpret_cast<const int4*>(Kh + (size_t)(t0 + tl) * hd + e0) : make_int4(0, 0, 0, 0);
      }
    }
    // the kUnroll positions' products, then their sums over the position's lanes level by
    // level, all positions at once (independent shuffles in flight together)
    unsigned long long dd[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      dd[u] = (unsigned long long)q0 * (unsigned long long)(long long)k4[u].x +
              (unsigned long long)q1 * (unsigned long long)(long long)k4[u].y +
              (unsigned long long)q2 * (unsigned long long)(long long)k4[u].z +
              (unsigned long long)q3 * (unsigned long long)(long long)k4[u].w;
    for (uint32_t o = lpp >> 1; o > 0; o >>= 1) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) dd[u] += __shfl_xor_sync(0xffffffffu, dd[u], o);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t tl = base + u * kWarps * ppw + slot;
      const unsigned long long d = dd[u];
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
  // the CTA's maximum goes into slot `rank` of every peer (thread r writes peer r); each CTA
  // then reads the maxima from its own shared memory once all have arrived
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  if (tid < CL) {
    long long mm = red[0];
    for (int w = 1; w < kWarps; ++w) mm = red[w] > mm ? red[w] : mm;
    st_async_peer(cmax + rank, (unsigned long long)mm, &xbar[0], tid);
  }
  exchange_wait(&xbar[0], p.state);
  long long m = LLONG_MIN;
  for (uint32_t r = 0; r < CL; ++r) m = cmax[r] > m ? cmax[r] : m;

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
  if (tid < CL) {
    unsigned long long t = 0;
    for (int w = 0; w < kWarps; ++w) t += (unsigned long long)red[w];
    st_async_peer(csum + rank, t, &xbar[1], tid);
  }
  // once this CTA's sums are in, nothing writes into its shared memory again (except in the
  // exchange of partial sums below, which has cluster barriers of its own)
  exchange_wait(&xbar[1], p.state);
  unsigned long long Z = 0;
  for (uint32_t r = 0; r < CL; ++r) Z += csum[r];

  // stage 2: P_t = (e_t << 24) / Z, 24 fractional bits
  const float rz = rcp_estimate((float)Z);  // Z >= 2^30: the largest score's entry is 2^30
  for (uint32_t tl = tid; tl < n; tl += kThreads)
    sc[tl] = (long long)div_by_estimate((unsigned long long)sc[tl] << 24, Z, rz);
  __syncthreads();

  // stage 3: sum over positions of P_t * v_t[j] (exact: |sum| < 2^55), then one >> 24
  unsigned long long a0 = 0, a1 = 0, a2 = 0, a3 = 0;
  cp_async_wait_all();  // the first batch of values
  for (uint32_t base = base0; base < n; base += kUnroll * kWarps * ppw) {
    int4 v4[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t tl = base + u * kWarps * ppw + slot;
      // first batch: slots past the chunk were never written, and their probability is 0
      v4[u] = base == base0 ? vpre[u * kThreads + tid]
              : tl < n      ? *reinterpret_cast<const int4*>(Vh + (size_t)(t0 + tl) * hd + e0)
                            : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t tl = base + u * kWarps * ppw + slot;
      const long long pr = tl < n ? sc[tl] : 0;
      a0 += (unsigned long long)(pr * (long long)v4[u].x);
      a1 += (unsigned long long)(pr * (long long)v4[u].y);
      a2 += (unsigned long long)(pr * (long long)v4[u].z);
      a3 += (unsigned long long)(pr * (long long)v4[u].w);
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
  if (p.o_acc) {
    // the CTA's partial sums go straight into the head's accumulators (wrapping adds, so the
    // order of the CTAs changes no bit); the next kernel applies the >> 24
    for (uint32_t j = tid; j < hd; j += kThreads) {
      unsigned long long s = 0;
      for (int w = 0; w < kWarps; ++w) s += part[(size_t)w * hd + j];
      atomicAdd(p.o_acc + (size_t)h * hd + j, s);
    }
    return;
  }
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
  return attn_vpre_offset(hd, chunk_cap) + (size_t)kUnroll * kThreads * 16;
}

// ------------------------------------------------------------------ long caches
// k_attention_long: the same four stages for caches whose chunks span many batches.  A copy
// warp streams the CTA's chunk of key rows, then of value rows, through a ring of
// shared-memory slots by bulk copies (a chunk of one head is one contiguous run: the cache is
// head-major), batch by batch, as soon as the consumers free a slot, so each SM has the ring's
// bytes in flight instead of the loads its threads can hold.  A batch is kLBatch bytes: 8192 /
// hd positions.  Scoring gives each lane NC chunks of 16 bytes of a key row (16 elements for
// heads of 16 or more), so a position's lane sums take few shuffle levels; the weighted sum of
// values gives each lane 4 elements (it needs no per-position sums).  Only the batch holding
// the newest row (written by the kernel just before) waits for that kernel; older rows stream
// at once.  The consumers exchange maxima and sums as in k_attention (remote stores that
// complete on the receiver's barrier); the copy warp takes no part and keeps streaming.
#ifndef CK_LSLOTS
#define CK_LSLOTS 5
#endif
#ifndef CK_LCLUSTER
#define CK_LCLUSTER 4
#endif
#ifndef CK_LLATE
#define CK_LLATE 1
#endif
constexpr uint32_t kLBatch = 32768;
constexpr uint32_t kLSlots = CK_LSLOTS;
constexpr int kLCluster = CK_LCLUSTER;  // CTAs a head: few enough that every cluster is resident at once
constexpr int kLWarps = 16;                    // consumer warps
constexpr int kLUnroll = 4;                    // warp steps of a value batch
constexpr int kLCons = kLWarps * 32;           // consumer threads
constexpr int kLThreads = kLCons + 32;         // + the copy warp
constexpr uint32_t kLPoll = 1u << 22;

// Shared memory of the long kernel: the ring, then the per-CTA region as k_attention lays it
// out (queries, partials, maximum, sum, reduction slots, scores), then the ring's barriers
// and the failure flag.
__host__ __device__ inline size_t lattn_region(uint32_t hd, uint32_t chunk_cap) {
  return 8 * ((size_t)hd * (2 + kLWarps) + 18 + kLWarps + chunk_cap);
}
__host__ __device__ inline size_t lattn_bars(uint32_t hd, uint32_t chunk_cap) {
  return ((size_t)kLSlots * kLBatch + lattn_region(hd, chunk_cap) + 15) & ~(size_t)15;
}
__host__ __device__ inline size_t lattn_smem(uint32_t hd, uint32_t chunk_cap) {
  return lattn_bars(hd, chunk_cap) + 2 * kLSlots * 8 + 16;
}

// A wait of the long kernel that ran out: the state is failed with error 9; the caller goes
// on without waiting, so that every thread reaches the same barriers.
__device__ __forceinline__ void lattn_fail(const AttnParams& p, volatile uint32_t* flag) {
  *flag = 1u;
  hdr<uint32_t>(p.state, kHError) = CK_CUDA_ERROR;
  hdr<uint32_t>(p.state, kHPhase) = CK_PHASE_FAILED;
}

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kLCons) : "memory"); }

template <int NC>
__global__ void __launch_bounds__(kLThreads, 1) k_attention_long(const AttnParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t hd = p.head_dim;
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* ring = smem;
  int64_t* q_s = reinterpret_cast<int64_t*>(smem + (size_t)kLSlots * kLBatch);
  unsigned long long* part = reinterpret_cast<unsigned long long*>(q_s + hd);  // [kLWarps][hd]
  unsigned long long* cpart = part + kLWarps * hd;                               // [hd]
  long long* cmax = reinterpret_cast<long long*>(cpart + hd);                   // [8], slot r from rank r
  unsigned long long* csum = reinterpret_cast<unsigned long long*>(cmax + 8);   // [8]
  uint64_t* xbar = reinterpret_cast<uint64_t*>(csum + 8);                        // [2]
  long long* red = reinterpret_cast<long long*>(xbar + 2);                      // [kLWarps]
  long long* sc = red + kLWarps;                                                 // [chunk_cap]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lattn_bars(hd, p.chunk_cap));
  uint64_t* empty = full + kLSlots;
  volatile uint32_t* flag = reinterpret_cast<volatile uint32_t*>(empty + kLSlots);

  const uint32_t pos = hdr_ld<uint32_t>(p.state, kHPosition);
  const uint32_t P = pos + 1;
  const uint32_t older = min(pos, p.cache);  // rows below this were written at earlier positions
  const uint32_t h = blockIdx.x;
  const uint32_t rank = cluster.block_rank(), CL = cluster.num_blocks();
  const uint32_t kvh = h / (p.heads / p.kv_heads);  // "head h reads key/value head h/(heads/kvHeads)"
  const uint32_t cs = (P + CL - 1) / CL;
  const uint32_t t0 = min(P, rank * cs), t1 = min(P, t0 + cs);
  const uint32_t n = t1 - t0;
  const int32_t* Kh = p.kcache + (size_t)kvh * p.cache * hd;
  const int32_t* Vh = p.vcache + (size_t)kvh * p.cache * hd;
  const uint32_t bp = kLBatch / (hd * 4);  // positions of a batch: SK warp steps of the keys,
                                           // kLUnroll of the values
  const uint32_t nb = (n + bp - 1) / bp;   // batches of keys (and of values)

  if (tid == 0) {
    for (uint32_t i = 0; i < kLSlots; ++i) {
      lbar_init(&full[i], 1);
      lbar_init(&empty[i], kLWarps);
    }
    for (int i = 0; i < 2; ++i) {  // the exchanges of maxima and sums: eight bytes from each CTA
      lbar_init(&xbar[i], 1);
      lbar_expect_tx(&xbar[i], 8 * CL);
    }
    *flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // every CTA has set up its barriers before a peer's first remote store into it (the
  // consumers wait on this arrival just before theirs)
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");

  if (warp == kLWarps) {
    // the copy warp: key batches, then value batches, into slot g % kLSlots for the g-th batch
    if (!CK_LLATE) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    uint32_t g = 0;
    bool waited = false, halt = false;
    auto issue = [&](const int32_t* base, uint32_t b) {
      const uint32_t slot = g % kLSlots;
      if (g >= kLSlots) {
        const uint32_t par = ((g / kLSlots) - 1) & 1u;
        uint32_t i = 0;
        while (!lbar_try(&empty[slot], par)) {
          if (*flag || ++i > kLPoll) {
            if (!*flag) lattn_fail(p, flag);
            halt = true;
            return;
          }
        }
      }
      const uint32_t r0 = b * bp, rows = min(bp, n - r0);
      if (!waited && t0 + r0 + rows > older) {  // the newest row: written by the kernel just before
        asm volatile("griddepcontrol.wait;" ::: "memory");
        waited = true;
      }
      lbar_expect_tx(&full[slot], rows * hd * 4);
      lbulk(ring + (size_t)slot * kLBatch, base + (size_t)(t0 + r0) * hd, rows * hd * 4, &full[slot]);
      ++g;
    };
    if (lane == 0) {
      for (uint32_t b = 0; b < nb && !halt; ++b) issue(Kh, b);
      for (uint32_t b = 0; b < nb && !halt; ++b) issue(Vh, b);  // as the consumers free slots
      // no copy outlives the CTA: the last kLSlots batches started have landed
      for (uint32_t j = g > kLSlots ? g - kLSlots : 0; j < g; ++j)
        for (uint32_t i = 0; i < kLPoll; ++i)
          if (lbar_try(&full[j % kLSlots], (j / kLSlots) & 1u)) break;
    }
    __syncwarp();
    if (CK_LLATE) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    return;
  }

  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!CK_LLATE) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const bool running = hdr_ld<uint32_t>(p.state, kHPhase) == CK_PHASE_RUNNING;
  for (uint32_t i = tid; i < hd; i += kLCons) q_s[i] = p.q[(size_t)h * hd + i];
  consumers_sync();
  // scoring: lane chunks j = 0..NC-1 of its 4 NC elements at rotated places, so that eight
  // consecutive lanes read eight different bank groups; the queries are permuted alike
  constexpr uint32_t E = 4 * NC, SH = NC == 4 ? 1 : NC == 2 ? 2 : 3, SK = 4 / NC;
  const uint32_t lppk = hd / E, ppwk = 32 / lppk;
  const uint32_t subk = lane % lppk, pslk = lane / lppk;
  uint32_t koff[NC];
  int64_t qp[NC][4];
#pragma unroll
  for (uint32_t j = 0; j < NC; ++j) {
    koff[j] = subk * E + 4 * ((j + (lane >> SH)) % NC);
#pragma unroll
    for (int e = 0; e < 4; ++e) qp[j][e] = q_s[koff[j] + e];
  }
  // weighted values: four elements a lane
  const uint32_t lpp = hd / 4, ppw = 32 / lpp;
  const uint32_t sub = lane % lpp, pslot = lane / lpp, e0 = sub * 4;
  bool dead = false;
  // a batch's slot, once its copies have landed (bounded; on a timeout the state fails)
  auto await = [&](uint32_t g) {
    if (dead) return;
    for (uint32_t i = 0; i < kLPoll; ++i) {
      if (lbar_try(&full[g % kLSlots], (g / kLSlots) & 1u)) return;
      if ((i & 63) == 63 && *flag) break;
    }
    if (!*flag) lattn_fail(p, flag);
    dead = true;
  };
  // an exchange's values, once the cluster's eight bytes a CTA have landed (bounded likewise)
  auto xwait = [&](uint64_t* bar) {
    for (uint32_t i = 0; i < kLPoll; ++i) {
      if (lbar_try(bar, 0)) return;
      if ((i & 63) == 63 && *flag) break;
    }
    if (!*flag) lattn_fail(p, flag);
    dead = true;
  };

  // stage 0: s_t = (((q . k_t) >> 16) * inv) >> 24, products and sums wrapping; keep the max
  long long lmax = LLONG_MIN;
  for (uint32_t b = 0; b < nb; ++b) {
    await(b);
    const int32_t* Kb = reinterpret_cast<const int32_t*>(ring + (size_t)(b % kLSlots) * kLBatch);
    unsigned long long dd[SK];
#pragma unroll
    for (uint32_t u = 0; u < SK; ++u) {
      const uint32_t tb = (u * kLWarps + warp) * ppwk + pslk, tl = b * bp + tb;
      unsigned long long a = 0;
#pragma unroll
      for (uint32_t j = 0; j < NC; ++j) {
        const int4 k = !dead && tl < n ? *reinterpret_cast<const int4*>(Kb + (size_t)tb * hd + koff[j])
                                       : make_int4(0, 0, 0, 0);
        a += (unsigned long long)qp[j][0] * (unsigned long long)(long long)k.x +
             (unsigned long long)qp[j][1] * (unsigned long long)(long long)k.y +
             (unsigned long long)qp[j][2] * (unsigned long long)(long long)k.z +
             (unsigned long long)qp[j][3] * (unsigned long long)(long long)k.w;
      }
      dd[u] = a;
    }
    for (uint32_t o = lppk >> 1; o > 0; o >>= 1) {  // all positions' lane sums at once
#pragma unroll
      for (uint32_t u = 0; u < SK; ++u) dd[u] += __shfl_xor_sync(0xffffffffu, dd[u], o);
    }
#pragma unroll
    for (uint32_t u = 0; u < SK; ++u) {
      const uint32_t tb = (u * kLWarps + warp) * ppwk + pslk, tl = b * bp + tb;
      const unsigned long long d = dd[u];
      if (tl < n && subk == 0) {
        long long sv = (long long)d >> 16;
        sv = (long long)((unsigned long long)sv * (unsigned long long)p.inv_sqrt) >> 24;
        sc[tl] = sv;
        lmax = sv > lmax ? sv : lmax;
      }
    }
    __syncwarp();
    if (lane == 0) lbar_arrive(&empty[b % kLSlots]);
  }
  lmax = warp_max(lmax);
  if (lane == 0) red[warp] = lmax;
  consumers_sync();
  // the CTA's maximum into slot `rank` of every peer (thread r writes peer r) by remote stores
  // that complete on the peer's barrier; the maxima are then read locally
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  if (tid < CL) {
    long long mm = red[0];
    for (int w = 1; w < kLWarps; ++w) mm = red[w] > mm ? red[w] : mm;
    st_async_peer(cmax + rank, (unsigned long long)mm, &xbar[0], tid);
  }
  xwait(&xbar[0]);
  long long m = LLONG_MIN;
  for (uint32_t r = 0; r < CL; ++r) m = cmax[r] > m ? cmax[r] : m;

  // stage 1: e_t = EXP[min((m - s_t) >> 8, 4096)]; the exact difference is >= 0 and fits u64
  unsigned long long z = 0;
  for (uint32_t tl = tid; tl < n; tl += kLCons) {
    unsigned long long idx = ((unsigned long long)m - (unsigned long long)sc[tl]) >> 8;
    if (idx > 4096) idx = 4096;
    const unsigned long long e = __ldg(p.exp_tab + idx);
    sc[tl] = (long long)e;
    z += e;
  }
  z = warp_sum(z);
  if (lane == 0) red[warp] = (long long)z;
  consumers_sync();
  if (tid < CL) {
    unsigned long long t = 0;
    for (int w = 0; w < kLWarps; ++w) t += (unsigned long long)red[w];
    st_async_peer(csum + rank, t, &xbar[1], tid);
  }
  xwait(&xbar[1]);  // after this nothing writes into this CTA's shared memory from outside
  unsigned long long Z = 0;
  for (uint32_t r = 0; r < CL; ++r) Z += csum[r];

  // stage 2: P_t = (e_t << 24) / Z, 24 fractional bits
  const float rz = rcp_estimate((float)Z);  // Z >= 2^30: the largest score's entry is 2^30
  for (uint32_t tl = tid; tl < n; tl += kLCons)
    sc[tl] = (long long)div_by_estimate((unsigned long long)sc[tl] << 24, Z, rz);
  consumers_sync();

  // stage 3: sum over positions of P_t * v_t[j] (exact: |sum| < 2^55), then one >> 24
  unsigned long long a0 = 0, a1 = 0, a2 = 0, a3 = 0;
  for (uint32_t b = 0; b < nb; ++b) {
    const uint32_t g = nb + b;
    await(g);
    const int32_t* Vb = reinterpret_cast<const int32_t*>(ring + (size_t)(g % kLSlots) * kLBatch);
#pragma unroll
    for (int u = 0; u < kLUnroll; ++u) {
      const uint32_t tb = (u * kLWarps + warp) * ppw + pslot, tl = b * bp + tb;
      if (!dead && tl < n) {
        const int4 v = *reinterpret_cast<const int4*>(Vb + (size_t)tb * hd + e0);
        const long long pr = sc[tl];
        a0 += (unsigned long long)(pr * (long long)v.x);
        a1 += (unsigned long long)(pr * (long long)v.y);
        a2 += (unsigned long long)(pr * (long long)v.z);
        a3 += (unsigned long long)(pr * (long long)v.w);
      }
    }
    __syncwarp();
    if (lane == 0) lbar_arrive(&empty[g % kLSlots]);
  }
  for (uint32_t o = 16; o >= lpp && o > 0; o >>= 1) {
    a0 += __shfl_xor_sync(0xffffffffu, a0, o);
    a1 += __shfl_xor_sync(0xffffffffu, a1, o);
    a2 += __shfl_xor_sync(0xffffffffu, a2, o);
    a3 += __shfl_xor_sync(0xffffffffu, a3, o);
  }
  if (pslot == 0) {
    unsigned long long* dst = part + (size_t)warp * hd + e0;
    dst[0] = a0;
    dst[1] = a1;
    dst[2] = a2;
    dst[3] = a3;
  }
  consumers_sync();
  // the next kernel's CTAs may start once this one's are finishing: launched earlier they
  // would hold SMs that clusters of this grid still wait for
  if (CK_LLATE) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the CTA's partial sums go straight into the head's accumulators (wrapping adds, so the
  // order of the CTAs changes no bit); the next kernel applies the >> 24
  if (running && *flag == 0u) {
    for (uint32_t j = tid; j < hd; j += kLCons) {
      unsigned long long sum = 0;
      for (int w = 0; w < kLWarps; ++w) sum += part[(size_t)w * hd + j];
      atomicAdd(p.o_acc + (size_t)h * hd + j, sum);
    }
  }
}

}  // namespace

int g_lattn_smem = 0;  // the opt-in shared memory of this device

cudaError_t configure_attention() {
  cudaError_t e = cudaFuncSetAttribute(k_attention, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
  int dev = 0, optin = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_attention_long<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_attention_long<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_attention_long<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e == cudaSuccess) g_lattn_smem = optin;
  return e;
}

#ifndef CK_LONG_BATCHES
#define CK_LONG_BATCHES 2
#endif
// The long-cache kernel takes heads whose chunks (over kLCluster CTAs) span more than this
// many batches, when the accumulator path is on and its shared memory fits.
uint32_t long_chunk(const AttnParams& p) { return (p.cache + kLCluster - 1) / kLCluster; }
bool attention_long(const AttnParams& p) {
  const uint32_t bp = kLBatch / (p.head_dim * 4);
  return p.o_acc && long_chunk(p) > CK_LONG_BATCHES * bp &&
         lattn_smem(p.head_dim, long_chunk(p)) <= (size_t)g_lattn_smem;
}

cudaError_t launch_attention(const AttnParams& p_in, cudaStream_t s, int cluster) {
  const bool lng = attention_long(p_in);
  AttnParams p = p_in;
  if (lng) {
    cluster = kLCluster;
    p.chunk_cap = long_chunk(p_in);
  }
  const size_t smem = lng ? lattn_smem(p.head_dim, p.chunk_cap) : attn_smem(p.head_dim, p.chunk_cap);
  if (!lng && smem > 96 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.heads, (unsigned)cluster, 1);
  cfg.blockDim = dim3(lng ? kLThreads : kThreads, 1, 1);
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
  if (!lng) return cudaLaunchKernelEx(&cfg, k_attention, p);
  if (p.head_dim >= 16) return cudaLaunchKernelEx(&cfg, k_attention_long<4>, p);
  if (p.head_dim == 8) return cudaLaunchKernelEx(&cfg, k_attention_long<2>, p);
  return cudaLaunchKernelEx(&cfg, k_attention_long<1>, p);
}

}  // namespace ck
