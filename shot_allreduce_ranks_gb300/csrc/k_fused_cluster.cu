// Fused LL8 packet allreduce whose per-owner scratch is the owner CTA's own
// shared memory, reached over the distributed shared memory of a
// thread-block cluster.
//
// The method is the monolithic fused packet allreduce of "Add monolithic
// fused packet allreduce kernel and Model::all_reduce_packet API"
// (microsoft/ark #254, Changes): every rank scatters the slices other ranks
// own as LL packets, each owner polls the packets' flags, reduces, and (write
// mode of "optimize allreduce write mode by broadcast output ptr",
// ROCm/aiter #1910, Motivation) stores the result straight into all R
// outputs.  On one GB300 the R virtual ranks of one chunk of the message are
// R CTAs of one cluster (cluster rank = virtual rank), so the packet slots an
// owner polls can live in that owner CTA's shared memory: producers write
// them with remote shared-memory stores, and the packets never reach L2 or
// HBM.  HBM then moves only the 4*R*N bytes of the one-shot minimum.
//
// Layout.  The groups of each rank's buffer are split into R shards of
// Vs = ceil(groups / R); rank o owns shard o.  Cluster c of C handles, in
// round k = 0..K-1, shard-local groups j = (k*C + c)*T + t (thread t of T).
// Owner o's ring in shared memory is [source slot (R-1)][T][4 packets]:
// thread t of producer s writes slot (s < o ? s : s-1), entry t, and only
// thread t of owner o reads it.
//
// One round, per thread: store the packets of round k (inputs loaded one
// round earlier) into the R-1 owners' rings; start the loads of round k+1;
// poll the own ring until the R-1 packet sets carry round k's flag, sum the
// R contributions in rank order 0..R-1 in fp32 (own input at position r),
// round once, store into all R outputs; then the cluster barrier
// (arrive.release / wait.acquire) orders every owner's reads of round k
// before any producer's stores of round k+1 into the same slots.
//
// Flags.  LL8 packet = 32-bit data word | 32-bit flag.  Round k of a call
// with device epoch e carries flag_at(e, k), the k-th value after e in the
// sequence that skips 0; the call moves the epoch on by K.  Each CTA zeroes
// its ring before a first cluster barrier, so leftover shared-memory
// contents never read as a flag.
//
// Waits.  A packet poll is bounded by the handle's spin limit (and an
// iteration cap); on expiry the thread records a timeout in the device error
// word and stops reducing for the rest of the call.  The cluster barriers
// are hardware barriers, not spins: every thread of every CTA of a cluster
// runs the same K + 1 of them (K depends only on the call's shape) and no
// thread leaves early, so each barrier completes; the last one also keeps
// every CTA's shared memory alive until no remote store can reach it.
#include "ar_internal.cuh"

namespace ar {
namespace {

constexpr int kClusterMaxThreads = 256;
constexpr uint32_t kClusterMaxSpins = 1u << 24;

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Address of the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
  return d;
}

__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_gpu_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// The four LL8 packets of one group into a remote CTA's ring entry: two
// 16-byte relaxed stores at cluster scope; each 64-bit packet is
// single-copy atomic, so a packet whose flag matches carries its data.
__device__ __forceinline__ void st_remote_packets(uint32_t addr, uint4 x, uint32_t flag) {
  const uint64_t hi = (uint64_t)flag << 32;
  asm volatile("st.relaxed.cluster.shared::cluster.v2.b64 [%0], {%1, %2};" ::"r"(addr),
               "l"(hi | x.x), "l"(hi | x.y)
               : "memory");
  asm volatile("st.relaxed.cluster.shared::cluster.v2.b64 [%0], {%1, %2};" ::"r"(addr + 16),
               "l"(hi | x.z), "l"(hi | x.w)
               : "memory");
}

__device__ __forceinline__ bool ld_local_packets(uint32_t addr, uint32_t flag, uint4& data) {
  uint64_t w0, w1, w2, w3;
  asm volatile("ld.relaxed.cluster.shared::cta.v2.b64 {%0, %1}, [%2];"
               : "=l"(w0), "=l"(w1)
               : "r"(addr)
               : "memory");
  asm volatile("ld.relaxed.cluster.shared::cta.v2.b64 {%0, %1}, [%2];"
               : "=l"(w2), "=l"(w3)
               : "r"(addr + 16)
               : "memory");
  data = make_uint4((uint32_t)w0, (uint32_t)w1, (uint32_t)w2, (uint32_t)w3);
  return (uint32_t)(w0 >> 32) == flag && (uint32_t)(w1 >> 32) == flag &&
         (uint32_t)(w2 >> 32) == flag && (uint32_t)(w3 >> 32) == flag;
}

__device__ __noinline__ void report_cluster_timeout(const FusedArgs& f, int owner, int source) {
  if (atomicCAS(&f.state->error, kDevErrNone, kDevErrTimeout) == kDevErrNone)
    f.state->error_info = ((uint32_t)owner << 16) | (uint32_t)source;
  atomicAdd(&f.state->timeouts, 1u);
}

// Bounded poll of one ring entry until its four packets carry `flag`.
__device__ __forceinline__ bool wait_local_packets(const FusedArgs& f, uint32_t addr,
                                                   uint32_t flag, uint4& data, int owner,
                                                   int source) {
  if (ld_local_packets(addr, flag, data)) return true;
  uint64_t t_first = 0;
  for (uint32_t spins = 1;; ++spins) {
    __nanosleep(16);
    if (ld_local_packets(addr, flag, data)) return true;
    if ((spins & 15u) == 0) {
      const uint64_t now = global_timer_ns();
      if (spins == 16u) t_first = now;
      if (spins > kClusterMaxSpins || (spins > 16u && now - t_first > f.spin_limit_ns)) {
        report_cluster_timeout(f, owner, source);
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t cluster_flag_at(uint32_t e, uint64_t k) {
  return (uint32_t)(((uint64_t)e - 1u + k) % 0xFFFFFFFFull + 1u);
}

// Input loads of shard-local group j: the R-1 groups other owners get from
// this rank (x[q-1] for owner (r+q) % R) and this rank's own group.
template <int R, class E>
__device__ __forceinline__ void load_round(const CallArgs& a, const char* my_in, int r, size_t Vs,
                                           size_t j, bool vec, uint64_t pol,
                                           uint4 (&x)[R > 1 ? R - 1 : 1], uint4& own) {
  if (j >= Vs) return;
#pragma unroll
  for (int q = 1; q < R; ++q) {
    const size_t g = (size_t)((r + q) % R) * Vs + j;
    if (g < a.groups) x[q - 1] = load_group<E, true>(my_in, g, group_valid<E>(g, a.count), vec, pol);
  }
  const size_t g = (size_t)r * Vs + j;
  if (g < a.groups) own = load_group<E, true>(my_in, g, group_valid<E>(g, a.count), vec, pol);
}

template <int R, class E>
__global__ void __launch_bounds__(kClusterMaxThreads, 2) k_fused_ll8_cluster(CallArgs a, FusedArgs f) {
  extern __shared__ __align__(16) uint64_t ring[];  // [R-1][T][4]
  __shared__ const char* s_in[R];
  __shared__ char* s_out[R];
  __shared__ uint32_t s_epoch;
  const int T = (int)blockDim.x, tid = (int)threadIdx.x;
  const int r = (int)cluster_ctarank();
  const size_t C = gridDim.x / R, c = blockIdx.x / R;
  const bool vec = load_tables<R>(a, s_in, s_out);
  if (tid == 0) s_epoch = ld_relaxed_gpu_u32(&f.state->epoch);
  for (int i = tid; i < (R - 1) * T * 4; i += T) ring[i] = 0ull;
  __syncthreads();
  cluster_barrier();  // every ring is zeroed before the first remote store

  const uint32_t epoch = s_epoch;
  const char* my_in = s_in[r];
  const size_t Vs = a.shard_groups;
  const size_t per_round = C * (size_t)T;
  const size_t K = (Vs + per_round - 1) / per_round;
  const uint64_t pol = l2_policy_evict_first();
  const uint32_t ring_base = smem_u32(ring);
  // My entry in the ring of owner (r + q) % R, and where source s lands in mine.
  uint32_t dst[R > 1 ? R - 1 : 1];
#pragma unroll
  for (int q = 1; q < R; ++q) {
    const int o = (r + q) % R;
    const int slot = r < o ? r : r - 1;
    dst[q - 1] = map_to_rank(ring_base + (uint32_t)((slot * T + tid) * 32), (uint32_t)o);
  }
  const bool produce = r != f.skip_producer;

  uint4 x[R > 1 ? R - 1 : 1];
  uint4 own = make_uint4(0, 0, 0, 0);
  const size_t j0 = c * (size_t)T + (size_t)tid;
  load_round<R, E>(a, my_in, r, Vs, j0, vec, pol, x, own);
  bool live = true;
  for (size_t k = 0; k < K; ++k) {
    const size_t j = k * per_round + j0;
    const uint32_t flag = cluster_flag_at(epoch, k);
    // ---- scatter round k into the owners' rings ----------------------------
    if (produce && j < Vs) {
#pragma unroll
      for (int q = 1; q < R; ++q) {
        const size_t g = (size_t)((r + q) % R) * Vs + j;
        if (g < a.groups) st_remote_packets(dst[q - 1], x[q - 1], flag);
      }
    }
    const uint4 own_k = own;
    // ---- loads of round k+1 are in flight while round k is reduced --------
    if (k + 1 < K) load_round<R, E>(a, my_in, r, Vs, j + per_round, vec, pol, x, own);
    // ---- poll + reduce + write-mode broadcast of round k ------------------
    const size_t g = (size_t)r * Vs + j;
    if (live && j < Vs && g < a.groups) {
      Acc<E> acc;
#pragma unroll
      for (int s = 0; s < R; ++s) {
        uint4 v = own_k;
        if (s != r && live) {
          const int slot = s < r ? s : s - 1;
          live = wait_local_packets(f, ring_base + (uint32_t)((slot * T + tid) * 32), flag, v, r, s);
        }
        if (s == 0) acc.set(v);
        else acc.add(v);
      }
      if (live) {
        const uint4 y = acc.round();
        const int valid = group_valid<E>(g, a.count);
#pragma unroll
        for (int q = 0; q < R; ++q) store_group<E>(s_out[q], g, y, valid, vec);
      }
    }
    __syncwarp();
    cluster_barrier();  // every owner has read round k before round k+1 is stored
  }

  // ---- flag rotation: the last CTA to finish moves the epoch on by K -------
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(&f.state->done, 1u);
    if (prev == gridDim.x - 1) {
      __threadfence();
      st_relaxed_gpu_u32(&f.state->done, 0u);
      st_relaxed_gpu_u32(&f.state->epoch, cluster_flag_at(epoch, K));
    }
  }
}

template <int R, class E>
cudaLaunchConfig_t cluster_config(LaunchCfg cfg, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)cfg.ctas);
  lc.blockDim = dim3((unsigned)cfg.threads);
  lc.dynamicSmemBytes = (size_t)(R - 1) * (size_t)cfg.threads * 32;
  lc.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = R;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return lc;
}

template <int R, class E>
cudaError_t cluster_prepare_impl() {
  return cudaFuncSetAttribute(k_fused_ll8_cluster<R, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (R - 1) * kClusterMaxThreads * 32);
}

template <int R, class E>
cudaError_t cluster_occ_impl(int threads, int* clusters) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t lc = cluster_config<R, E>({R * 64, threads}, nullptr, attr);
  return cudaOccupancyMaxActiveClusters(clusters, k_fused_ll8_cluster<R, E>, &lc);
}

template <int R, class E>
cudaError_t cluster_launch_impl(const CallArgs& a, const FusedArgs& f, LaunchCfg cfg,
                                cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t lc = cluster_config<R, E>(cfg, s, attr);
  return cudaLaunchKernelEx(&lc, k_fused_ll8_cluster<R, E>, a, f);
}

}  // namespace

cudaError_t cluster_prepare(int R, int dtype) {
#define P(RR, EE) return cluster_prepare_impl<RR, EE>()
  AR_DISPATCH(dtype, R, P, AR_SWITCH_R8)
#undef P
  return cudaErrorInvalidValue;
}

static cudaError_t cluster_occ(int R, int dtype, int threads, int* n) {
#define Q(RR, EE) return cluster_occ_impl<RR, EE>(threads, n)
  AR_DISPATCH(dtype, R, Q, AR_SWITCH_R8)
#undef Q
  return cudaErrorInvalidValue;
}

int cluster_max_active(int R, int dtype, int threads) {
  if (threads < 32 || threads > kClusterMaxThreads || threads % 32) return 0;
  int n = 0;
  if (cluster_occ(R, dtype, threads, &n) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_fused_ll8_cluster(int R, int dtype, const CallArgs& a, const FusedArgs& f,
                                     LaunchCfg cfg, cudaStream_t s) {
  if (cfg.ctas % R != 0 || cfg.threads > kClusterMaxThreads || cfg.threads % 32)
    return cudaErrorInvalidValue;
#define L(RR, EE) return cluster_launch_impl<RR, EE>(a, f, cfg, s)
  AR_DISPATCH(dtype, R, L, AR_SWITCH_R8)
#undef L
  return cudaErrorInvalidValue;
}

}  // namespace ar
