// One-shot fan-out (write mode) with the data moved by the bulk-copy (TMA)
// engine instead of per-thread loads.
//
// Same result and the same 4*R*N bytes as k_oneshot_fanout ("One shot all
// reduce Example", pytorch-labs/helion #245, read of all ranks; "optimize
// allreduce write mode by broadcast output ptr", ROCm/aiter #1910,
// Motivation: the reduced data written straight into every rank's output).
// What changes is how the bytes get in flight: a persistent CTA keeps S tiles
// of all R inputs in a shared-memory ring, filled by cp.async.bulk copies
// that complete on one mbarrier per stage, so the number of bytes in flight
// no longer depends on registers.  Threads sum a tile from shared memory in
// rank order, round once, write the result tile to shared memory, and one
// thread sends it to all R outputs with R bulk stores.
//
// Tile = 256 threads x 16 bytes = 4 KiB per rank.  Tile t covers bytes
// [4096 t, 4096 t + 4096) of every rank; CTA b takes tiles b, b + G, ...
// Only whole 16-byte groups go through tiles (bulk copies move multiples of
// 16 bytes); the last partial group is summed by the last CTA with
// element-sized accesses.  A call whose pointers are not all 16-byte aligned
// runs the element path in every CTA.
//
// Every wait on an mbarrier is bounded by the handle's spin limit; on expiry
// the CTA records kDevErrCopyTimeout, waits (bounded again) for the copies it
// still has in flight, and returns.
#include "ar_internal.cuh"

namespace ar {
namespace {

constexpr uint32_t kTileBytes = kBulkThreads * kGroupBytes;  // 4096
constexpr int kTileGroups = kBulkThreads;                     // one group per thread

// Stages of the input ring: about 128 KiB of tiles in flight per CTA.
template <int R>
__host__ __device__ constexpr int bulk_stages() {
  return (128 * 1024) / (R * (int)kTileBytes) < 2 ? 2
         : (128 * 1024) / (R * (int)kTileBytes) > 8 ? 8
                                                    : (128 * 1024) / (R * (int)kTileBytes);
}

template <int R>
__host__ __device__ constexpr size_t bulk_smem() {
  return (size_t)bulk_stages<R>() * R * kTileBytes + 2 * kTileBytes;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t k = 0; k < (1u << 26); ++k) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((k & 63u) == 63u && global_timer_ns() - t0 > limit_ns) return false;
  }
  return false;
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_addr(src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 lds_v4(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

__device__ __forceinline__ void sts_v4(void* p, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(smem_addr(p)), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __noinline__ void report_copy_timeout(DevState* st) {
  if (atomicCAS(&st->error, kDevErrNone, kDevErrCopyTimeout) == kDevErrNone)
    st->error_info = 0xFFFF0000u | (blockIdx.x & 0xFFFFu);
  atomicAdd(&st->timeouts, 1u);
}

// Whole groups of tile t (the tiles cover `full` groups).
__device__ __forceinline__ uint32_t bulk_tile_groups(size_t t, size_t full) {
  const size_t left = full - t * kTileGroups;
  return left < (size_t)kTileGroups ? (uint32_t)left : (uint32_t)kTileGroups;
}

// Thread 0: start the R bulk loads of this CTA's i-th tile into stage i % S.
template <int R, int S>
__device__ __forceinline__ void bulk_issue(uint8_t* in_tiles, const char* const* s_in,
                                           uint64_t* full, size_t i, size_t nfull, uint64_t pol) {
  const size_t t = (size_t)blockIdx.x + i * gridDim.x;
  const int s = (int)(i % S);
  const uint32_t bytes = bulk_tile_groups(t, nfull) * (uint32_t)kGroupBytes;
  mbar_arrive_expect_tx(&full[s], bytes * R);
#pragma unroll
  for (int r = 0; r < R; ++r)
    bulk_load(in_tiles + ((size_t)s * R + r) * kTileBytes, s_in[r] + t * kTileBytes, bytes,
              &full[s], pol);
}

template <int R, class E>
__global__ void __launch_bounds__(kBulkThreads) k_oneshot_fanout_bulk(CallArgs a) {
  constexpr int S = bulk_stages<R>();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[S];
  __shared__ const char* s_in[R];
  __shared__ char* s_out[R];
  // The caller's pointer tables are read before waiting for the previous
  // kernel in the stream (programmatic dependent launch), so that round trip
  // overlaps its tail; inputs and outputs are touched only after the wait.
  const bool vec = load_tables<R>(a, s_in, s_out);
  pdl_enter();
  const int tid = threadIdx.x;

  if (!vec) {  // element path: some pointer is not 16-byte aligned
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t g = (size_t)blockIdx.x * blockDim.x + tid; g < a.groups; g += stride) {
      const int valid = group_valid<E>(g, a.count);
      uint4 x[R];
#pragma unroll
      for (int s = 0; s < R; ++s) x[s] = load_group<E>(s_in[s], g, valid, false);
      Acc<E> acc;
      acc.set(x[0]);
#pragma unroll
      for (int s = 1; s < R; ++s) acc.add(x[s]);
      const uint4 y = acc.round();
#pragma unroll
      for (int r = 0; r < R; ++r) store_group<E>(s_out[r], g, y, valid, false);
    }
    return;
  }

  uint8_t* in_tiles = smem;                               // [S][R][kTileBytes]
  uint8_t* res_tiles = smem + (size_t)S * R * kTileBytes;  // [2][kTileBytes]
  const size_t nfull = a.count / E::kGroup;  // whole groups
  const size_t ntiles = (nfull + kTileGroups - 1) / kTileGroups;
  const size_t my_n =
      blockIdx.x < ntiles ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const uint64_t pol = l2_policy_evict_first();
  if (tid == 0)
    for (size_t i = 0; i < my_n && i < (size_t)S; ++i)
      bulk_issue<R, S>(in_tiles, s_in, full, i, nfull, pol);

  size_t i = 0;
  for (; i < my_n; ++i) {
    const int s = (int)(i % S);
    const uint32_t parity = (uint32_t)((i / S) & 1);
    const size_t t = (size_t)blockIdx.x + i * gridDim.x;
    const uint32_t groups = bulk_tile_groups(t, nfull);
    const bool ok = mbar_wait_bounded(&full[s], parity, a.spin_limit_ns);
    if (tid == 0) bulk_wait_read<1>();  // stores of tile i-2 have read res[i & 1]
    if (__syncthreads_or(!ok)) break;
    uint8_t* res = res_tiles + (i & 1) * kTileBytes;
    if ((uint32_t)tid < groups) {
      const uint8_t* base = in_tiles + (size_t)s * R * kTileBytes + (size_t)tid * kGroupBytes;
      uint4 x[R];
#pragma unroll
      for (int r = 0; r < R; ++r) x[r] = lds_v4(base + (size_t)r * kTileBytes);
      Acc<E> acc;
      acc.set(x[0]);
#pragma unroll
      for (int r = 1; r < R; ++r) acc.add(x[r]);
      sts_v4(res + (size_t)tid * kGroupBytes, acc.round());
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      const uint32_t bytes = groups * (uint32_t)kGroupBytes;
#pragma unroll
      for (int r = 0; r < R; ++r) bulk_store(s_out[r] + t * kTileBytes, res, bytes);
      bulk_commit();
      if (i + S < my_n) bulk_issue<R, S>(in_tiles, s_in, full, i + S, nfull, pol);
    }
  }

  if (i < my_n) {
    // A copy wait ran out: record it, then give the copies still in flight
    // (tiles i .. min(i + S, my_n) - 1) one more bounded chance to land
    // before the CTA's shared memory goes away.
    if (tid == 0) {
      report_copy_timeout(a.state);
      for (size_t k = i; k < my_n && k < i + S; ++k)
        mbar_wait_bounded(&full[k % S], (uint32_t)((k / S) & 1), a.spin_limit_ns);
    }
    __syncthreads();
  }
  if (tid == 0) bulk_wait<0>();

  // The elements of the last, partial group.
  const size_t first_tail = nfull * E::kGroup;
  if (blockIdx.x == gridDim.x - 1 && (size_t)tid < a.count - first_tail) {
    const size_t off = (first_tail + tid) * E::kBytes;
    float acc = E::to_f32(ld_elem<E::kBytes>(s_in[0] + off));
#pragma unroll
    for (int r = 1; r < R; ++r) acc = __fadd_rn(acc, E::to_f32(ld_elem<E::kBytes>(s_in[r] + off)));
    const uint32_t y = E::from_f32(acc);
#pragma unroll
    for (int r = 0; r < R; ++r) st_elem<E::kBytes>(s_out[r] + off, y);
  }
}

}  // namespace

size_t bulk_smem_bytes(int R) {
  switch (R) {
#define B(RR) \
  case RR:    \
    return bulk_smem<RR>();
    B(1) B(2) B(3) B(4) B(5) B(6) B(7) B(8) B(9) B(10) B(11) B(12) B(13) B(14) B(15) B(16)
#undef B
    default:
      return 0;
  }
}

cudaError_t bulk_prepare(int R, int dtype) {
#define P(RR, EE)                                                                   \
  return cudaFuncSetAttribute(k_oneshot_fanout_bulk<RR, EE>,                        \
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bulk_smem<RR>())
  AR_DISPATCH(dtype, R, P, AR_SWITCH_R16)
#undef P
  return cudaErrorInvalidValue;
}

static cudaError_t bulk_occ(int R, int dtype, int* n) {
#define Q(RR, EE)                                                                              \
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, k_oneshot_fanout_bulk<RR, EE>,       \
                                                       kBulkThreads, bulk_smem<RR>())
  AR_DISPATCH(dtype, R, Q, AR_SWITCH_R16)
#undef Q
  return cudaErrorInvalidValue;
}

int bulk_ctas_per_sm(int R, int dtype) {
  int n = 0;
  return bulk_occ(R, dtype, &n) == cudaSuccess ? n : 0;
}

cudaError_t launch_oneshot_fanout_bulk(int R, int dtype, const CallArgs& a, LaunchCfg cfg,
                                       cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cfg.threads = kBulkThreads;
#define L(RR, EE)                                                                             \
  {                                                                                           \
    const cudaLaunchConfig_t lc = plain_config(cfg, dim3((unsigned)cfg.ctas), bulk_smem<RR>(), s, \
                                               attr);                                         \
    return cudaLaunchKernelEx(&lc, k_oneshot_fanout_bulk<RR, EE>, a);                         \
  }
  AR_DISPATCH(dtype, R, L, AR_SWITCH_R16)
#undef L
  return cudaErrorInvalidValue;
}

}  // namespace ar
