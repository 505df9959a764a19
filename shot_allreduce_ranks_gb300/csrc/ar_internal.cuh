// Internal declarations shared by the library's CUDA translation units.
// Device helpers are header-only (static inline) so no device linking is
// needed; every kernel is instantiated for a compile-time rank count R.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ar.h"

namespace ar {

constexpr int kVecElems = 8;  // bf16 elements per 16-byte vector ("group")

// ---------------------------------------------------------------------------
// Device-resident state of one handle (one per handle, 64 bytes).
struct DevState {
  uint32_t epoch;       // LL8 flag of the next fused call, in [1, 2^32-1]
  uint32_t done;        // CTAs of the running fused call that have finished
  uint32_t error;       // 0, or a DevError code (first error wins)
  uint32_t error_info;  // (waiting rank << 16) | missing source rank of the first timeout
  uint32_t timeouts;    // number of packet waits that gave up
  uint32_t abort_epoch; // epoch of the last call abandoned after a timeout
  uint32_t pad[10];
};

// Device error codes.  kDevErrTimeout: an LL8 packet wait gave up.
// kDevErrCopyTimeout: a wait for a bulk (TMA) copy into shared memory gave up.
enum DevError : uint32_t { kDevErrNone = 0, kDevErrTimeout = 1, kDevErrCopyTimeout = 2 };

// Everything a kernel needs about one call, passed by value.
struct CallArgs {
  const uint16_t* const* in_tbl;  // device array of R input pointers
  uint16_t* const* out_tbl;       // device array of R output pointers
  size_t count;                   // elements per rank
  size_t groups;                  // ceil(count / 8)
  size_t shard_groups;            // ceil(groups / R): groups owned by each rank
  DevState* state;                // the handle's state block (error word)
  uint64_t spin_limit_ns;         // bound of every device-side wait
};

// Extra arguments of the fused packet kernel.
struct FusedArgs {
  uint64_t* scratch;      // packets, layout [owner][source slot][group][4]
  uint64_t* rscratch;     // result packets of the staged variants, [dest][owner slot][group][4]
  size_t slot_groups;     // groups per (owner, source) slot = shard_groups at max_count
  DevState* state;
  uint64_t spin_limit_ns;
  int skip_producer;      // test hook: rank whose packet stores are skipped, or -1
  // Ring variant only: packets live in `scratch` as a ring of ring_depth
  // rounds per (owner, source, CTA); progress[(owner, c, warp)] is the flag
  // of the last round that warp of CTA c of `owner` finished reading.
  int ring_depth;
  uint32_t* progress;
};

constexpr int kMaxRingCtas = 1024;  // CTAs per rank the ring progress array can hold
constexpr int kMaxRingWarps = 16;   // warps per CTA (512 threads)
constexpr int kMaxRingDepth = 4;
// Progress words per rank: one per (CTA, warp).
constexpr size_t kRingProgressWords = (size_t)kMaxRingCtas * kMaxRingWarps;

// ---------------------------------------------------------------------------
// Small device helpers.

// 16-byte global accesses that bypass L1 allocation.  With kHint the access
// carries an L2 cache policy (createpolicy) chosen by the caller.
template <bool kHint = false>
__device__ __forceinline__ uint4 ld_v4_stream(const uint16_t* p, uint64_t pol = 0) {
  uint4 v;
  if (kHint) {
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
  } else {
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
  }
  return v;
}

template <bool kHint = false>
__device__ __forceinline__ void st_v4_stream(uint16_t* p, uint4 v, uint64_t pol = 0) {
  if (kHint) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
  } else {
    asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
  }
}

// L2 policy under which a line is among the first to be evicted (data that
// streams through once).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint16_t ld_u16(const uint16_t* p) {
  unsigned short v;
  asm volatile("ld.global.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_u16(uint16_t* p, uint16_t v) {
  asm volatile("st.global.u16 [%0], %1;" ::"l"(p), "h"((unsigned short)v) : "memory");
}

// Load group g (8 elements) of a buffer.  `valid` < 8 only for the last,
// partial group; `vec` is false when some pointer of the call is not
// 16-byte aligned.  Missing elements read as +0 (never stored back).
template <bool kHint = false>
__device__ __forceinline__ uint4 load_group(const uint16_t* base, size_t g, int valid, bool vec,
                                            uint64_t pol = 0) {
  const uint16_t* p = base + g * kVecElems;
  if (vec && valid == kVecElems) return ld_v4_stream<kHint>(p, pol);
  uint32_t w0 = 0u, w1 = 0u, w2 = 0u, w3 = 0u;
#pragma unroll
  for (int e = 0; e < kVecElems; ++e) {
    if (e < valid) {
      const uint32_t h = (uint32_t)ld_u16(p + e) << (16 * (e & 1));
      if (e < 2) w0 |= h;
      else if (e < 4) w1 |= h;
      else if (e < 6) w2 |= h;
      else w3 |= h;
    }
  }
  return make_uint4(w0, w1, w2, w3);
}

template <bool kHint = false>
__device__ __forceinline__ void store_group(uint16_t* base, size_t g, uint4 v, int valid, bool vec,
                                            uint64_t pol = 0) {
  uint16_t* p = base + g * kVecElems;
  if (vec && valid == kVecElems) {
    st_v4_stream<kHint>(p, v, pol);
    return;
  }
#pragma unroll
  for (int e = 0; e < kVecElems; ++e) {
    if (e < valid) {
      const uint32_t w = e < 2 ? v.x : e < 4 ? v.y : e < 6 ? v.z : v.w;
      st_u16(p + e, (uint16_t)(w >> (16 * (e & 1))));
    }
  }
}

// bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32 word.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> one word of two bf16, each rounded to nearest even
// (cvt.rn.bf16x2.f32 puts its first source in the upper half).
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Eight fp32 accumulators for one group.
struct Acc8 {
  float v[8];
  __device__ __forceinline__ void set(uint4 x) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = bf16_lo(w[k]);
      v[2 * k + 1] = bf16_hi(w[k]);
    }
  }
  // One rank-order step: acc = acc + x (plain fp32 add, round to nearest).
  __device__ __forceinline__ void add(uint4 x) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __fadd_rn(v[2 * k], bf16_lo(w[k]));
      v[2 * k + 1] = __fadd_rn(v[2 * k + 1], bf16_hi(w[k]));
    }
  }
  __device__ __forceinline__ uint4 round_bf16() const {
    return make_uint4(pack_bf16x2_rn(v[0], v[1]), pack_bf16x2_rn(v[2], v[3]),
                      pack_bf16x2_rn(v[4], v[5]), pack_bf16x2_rn(v[6], v[7]));
  }
};

// Number of valid elements in group g of a buffer of `count` elements.
__device__ __forceinline__ int group_valid(size_t g, size_t count) {
  const size_t first = g * kVecElems;
  const size_t left = count - first;
  return left >= (size_t)kVecElems ? kVecElems : (int)left;
}

// Copy the R input and output pointers of a call into shared memory, and
// decide (CTA-uniformly) whether every pointer allows 16-byte vectors.
template <int R>
__device__ __forceinline__ bool load_tables(const CallArgs& a, const uint16_t** s_in, uint16_t** s_out) {
  __shared__ int s_misaligned;
  if (threadIdx.x == 0) s_misaligned = 0;
  __syncthreads();
  if (threadIdx.x < R) {
    const uint16_t* p = a.in_tbl[threadIdx.x];
    s_in[threadIdx.x] = p;
    if (reinterpret_cast<uintptr_t>(p) & 15u) atomicOr(&s_misaligned, 1);
  } else if (threadIdx.x < 2 * R) {
    uint16_t* p = a.out_tbl[threadIdx.x - R];
    s_out[threadIdx.x - R] = p;
    if (reinterpret_cast<uintptr_t>(p) & 15u) atomicOr(&s_misaligned, 1);
  }
  __syncthreads();
  return s_misaligned == 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// Host-side launch descriptions.

struct LaunchCfg {
  int ctas;
  int threads;
};

// Launchers (defined in the kernel translation units).  Each returns the
// CUDA error of its launch(es).
cudaError_t launch_oneshot_pull(int R, const CallArgs& a, LaunchCfg cfg, cudaStream_t s);
cudaError_t launch_oneshot_fanout(int R, const CallArgs& a, LaunchCfg cfg, cudaStream_t s);
cudaError_t launch_twophase(int R, const CallArgs& a, LaunchCfg cfg, cudaStream_t s);
cudaError_t launch_fused_ll8(int R, const CallArgs& a, const FusedArgs& f, LaunchCfg cfg,
                             cudaStream_t s);
cudaError_t launch_fused_ll8_staged(int R, const CallArgs& a, const FusedArgs& f, LaunchCfg cfg,
                                    cudaStream_t s);
cudaError_t launch_packet_3op(int R, const CallArgs& a, const FusedArgs& f, LaunchCfg cfg,
                              cudaStream_t s);
int fused_staged_ctas_per_sm(int R, int threads);
cudaError_t launch_fused_ll8_ring(int R, const CallArgs& a, const FusedArgs& f, LaunchCfg cfg,
                                  cudaStream_t s);
int fused_ring_ctas_per_sm(int R, int threads);
// Reduce-scatter / all-gather (k_rs_ag.cu): a.count is the block length;
// the grid is (cfg.ctas, R).
cudaError_t launch_reduce_scatter(int R, const CallArgs& a, LaunchCfg cfg, cudaStream_t s);
cudaError_t launch_all_gather(int R, const CallArgs& a, LaunchCfg cfg, cudaStream_t s);

// Occupancy (CTAs per SM) of the fused and fan-out kernels for R ranks and
// `threads` threads per CTA.
int fused_ctas_per_sm(int R, int threads);
int fanout_ctas_per_sm(int R, int threads);

// Bulk-copy fan-out (k_oneshot_bulk.cu): fixed 256 threads per CTA, dynamic
// shared memory per CTA, CTAs per SM, and a one-time attribute set-up.
constexpr int kBulkThreads = 256;
size_t bulk_smem_bytes(int R);
int bulk_ctas_per_sm(int R);
cudaError_t bulk_prepare(int R);
cudaError_t launch_oneshot_fanout_bulk(int R, const CallArgs& a, int ctas, cudaStream_t s);

}  // namespace ar

// Expands CALL(1) .. CALL(8) on a runtime rank count inside a launcher that
// returns cudaError_t.
#define AR_RANK_SWITCH(R, CALL)            \
  switch (R) {                             \
    case 1: CALL(1); break;                \
    case 2: CALL(2); break;                \
    case 3: CALL(3); break;                \
    case 4: CALL(4); break;                \
    case 5: CALL(5); break;                \
    case 6: CALL(6); break;                \
    case 7: CALL(7); break;                \
    case 8: CALL(8); break;                \
    default: return cudaErrorInvalidValue; \
  }
