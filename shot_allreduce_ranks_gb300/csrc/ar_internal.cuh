// Internal declarations shared by the library's CUDA translation units.
// Device helpers are header-only (static inline) so no device linking is
// needed; every kernel is instantiated for a compile-time rank count R and
// element type E.  Data moves in 16-byte "groups": 8 bf16, 8 fp16 or 4 fp32
// elements; an LL8 packet carries one 32-bit word of a group.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ar.h"

namespace ar {

constexpr int kGroupBytes = 16;  // bytes per vector access ("group")

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
  const char* const* in_tbl;      // device array of R input pointers
  char* const* out_tbl;           // device array of R output pointers
  size_t count;                   // elements per rank
  size_t groups;                  // ceil(count / elements per group)
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
  // Write-mode fused kernel only.  lead: tiles a CTA scatters ahead of the
  // tile it reduces (>= 1).  discard: drop consumed packet lines from L2
  // without writing them back (set only where the scratch's memory contents
  // are known to hold zeros or older packets, see ar_create).
  int lead;
  int discard;
  int fast32;   // every slot and input group offset of the call fits in 32 bits
  // Ring mode of the write-mode fused kernel (ring_rounds > 0): every CTA
  // keeps its packets in a private ring of ring_rounds rounds in `ring`
  // ([CTA][round slot][owner][source slot][Tr groups][4]) instead of the
  // message-sized scratch, and reuses a slot after a CTA barrier.
  uint64_t* ring;
  int ring_rounds;
  // Test hook: CTAs of virtual rank delay_rank (or none if -1) wait delay_ns
  // of %globaltimer before their first packet store (a skewed producer).
  int delay_rank;
  uint64_t delay_ns;
};

// ---------------------------------------------------------------------------
// Small device helpers.

// 16-byte global accesses that bypass L1 allocation.  With kHint the access
// carries an L2 cache policy (createpolicy) chosen by the caller.
template <bool kHint = false>
__device__ __forceinline__ uint4 ld_v4_stream(const char* p, uint64_t pol = 0) {
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
__device__ __forceinline__ void st_v4_stream(char* p, uint4 v, uint64_t pol = 0) {
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

// ---------------------------------------------------------------------------
// Element types.  Each gives the elements per group, the element size, and
// exact widening to fp32 / round-to-nearest-even narrowing from fp32 of one
// element's bits.  Widening is exact for all three; fp32 is not rounded.

__device__ __forceinline__ uint32_t cvt_rn_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));  // first source -> upper half
  return d;
}

__device__ __forceinline__ uint32_t cvt_rn_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float cvt_f32_f16(uint32_t h) {
  float f;
  const unsigned short hs = (unsigned short)h;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(hs));
  return f;
}

struct Bf16 {
  static constexpr int kGroup = 8;
  static constexpr int kBytes = 2;
  __device__ static float lo(uint32_t w) { return __uint_as_float(w << 16); }
  __device__ static float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
  __device__ static uint32_t pack(float lo, float hi) { return cvt_rn_bf16x2(lo, hi); }
  __device__ static float to_f32(uint32_t bits) { return __uint_as_float(bits << 16); }
  __device__ static uint32_t from_f32(float x) { return cvt_rn_bf16x2(x, 0.0f) & 0xFFFFu; }
};

struct F16 {
  static constexpr int kGroup = 8;
  static constexpr int kBytes = 2;
  __device__ static float lo(uint32_t w) { return cvt_f32_f16(w & 0xFFFFu); }
  __device__ static float hi(uint32_t w) { return cvt_f32_f16(w >> 16); }
  __device__ static uint32_t pack(float lo, float hi) { return cvt_rn_f16x2(lo, hi); }
  __device__ static float to_f32(uint32_t bits) { return cvt_f32_f16(bits); }
  __device__ static uint32_t from_f32(float x) { return cvt_rn_f16x2(x, 0.0f) & 0xFFFFu; }
};

struct F32 {
  static constexpr int kGroup = 4;
  static constexpr int kBytes = 4;
  __device__ static float to_f32(uint32_t bits) { return __uint_as_float(bits); }
  __device__ static uint32_t from_f32(float x) { return __float_as_uint(x); }
};

// Accumulators for one group: the rank-order fp32 sum of its elements.
template <class E>
struct Acc;

template <class E>
struct AccHalf {  // bf16 / fp16: two elements per 32-bit word
  float v[8];
  __device__ __forceinline__ void set(uint4 x) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = E::lo(w[k]);
      v[2 * k + 1] = E::hi(w[k]);
    }
  }
  // One rank-order step: acc = acc + x (plain fp32 add, round to nearest).
  __device__ __forceinline__ void add(uint4 x) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __fadd_rn(v[2 * k], E::lo(w[k]));
      v[2 * k + 1] = __fadd_rn(v[2 * k + 1], E::hi(w[k]));
    }
  }
  __device__ __forceinline__ uint4 round() const {
    return make_uint4(E::pack(v[0], v[1]), E::pack(v[2], v[3]), E::pack(v[4], v[5]),
                      E::pack(v[6], v[7]));
  }
};

template <>
struct Acc<Bf16> : AccHalf<Bf16> {};
template <>
struct Acc<F16> : AccHalf<F16> {};

template <>
struct Acc<F32> {
  float v[4];
  __device__ __forceinline__ void set(uint4 x) {
    v[0] = __uint_as_float(x.x);
    v[1] = __uint_as_float(x.y);
    v[2] = __uint_as_float(x.z);
    v[3] = __uint_as_float(x.w);
  }
  __device__ __forceinline__ void add(uint4 x) {
    v[0] = __fadd_rn(v[0], __uint_as_float(x.x));
    v[1] = __fadd_rn(v[1], __uint_as_float(x.y));
    v[2] = __fadd_rn(v[2], __uint_as_float(x.z));
    v[3] = __fadd_rn(v[3], __uint_as_float(x.w));
  }
  __device__ __forceinline__ uint4 round() const {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                      __float_as_uint(v[3]));
  }
};

// Packed pairs of fp32 values (low element in the low 32 bits) and their
// IEEE round-to-nearest-even addition, one instruction for both lanes.  Each
// lane is exactly a plain fp32 add (no flush of subnormals), so a sum built
// from these is bit-identical to one built from scalar adds in the same order.
__device__ __forceinline__ uint64_t f32x2_make(uint32_t lo_bits, uint32_t hi_bits) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo_bits), "r"(hi_bits));
  return d;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ void f32x2_split(uint64_t p, float& lo, float& hi) {
  uint32_t a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(a), "=r"(b) : "l"(p));
  lo = __uint_as_float(a);
  hi = __uint_as_float(b);
}

// The rank-order accumulator of one group kept as packed pairs: same
// results as Acc<E>, half the add instructions.
template <class E>
struct Acc2 {  // bf16 / fp16: word k of a group holds elements 2k (low) and 2k+1
  uint64_t v[4];
  __device__ __forceinline__ static uint64_t widen(uint32_t w) {
    return f32x2_make(__float_as_uint(E::lo(w)), __float_as_uint(E::hi(w)));
  }
  __device__ __forceinline__ void set(uint4 x) {
    v[0] = widen(x.x);
    v[1] = widen(x.y);
    v[2] = widen(x.z);
    v[3] = widen(x.w);
  }
  __device__ __forceinline__ void add(uint4 x) {
    v[0] = f32x2_add(v[0], widen(x.x));
    v[1] = f32x2_add(v[1], widen(x.y));
    v[2] = f32x2_add(v[2], widen(x.z));
    v[3] = f32x2_add(v[3], widen(x.w));
  }
  __device__ __forceinline__ uint4 round() const {
    float a[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) f32x2_split(v[k], a[2 * k], a[2 * k + 1]);
    return make_uint4(E::pack(a[0], a[1]), E::pack(a[2], a[3]), E::pack(a[4], a[5]),
                      E::pack(a[6], a[7]));
  }
};

template <>
struct Acc2<F32> {  // four fp32 elements: two pairs
  uint64_t v[2];
  __device__ __forceinline__ void set(uint4 x) {
    v[0] = f32x2_make(x.x, x.y);
    v[1] = f32x2_make(x.z, x.w);
  }
  __device__ __forceinline__ void add(uint4 x) {
    v[0] = f32x2_add(v[0], f32x2_make(x.x, x.y));
    v[1] = f32x2_add(v[1], f32x2_make(x.z, x.w));
  }
  __device__ __forceinline__ uint4 round() const {
    uint32_t a, b, c, d;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(a), "=r"(b) : "l"(v[0]));
    asm("mov.b64 {%0, %1}, %2;" : "=r"(c), "=r"(d) : "l"(v[1]));
    return make_uint4(a, b, c, d);
  }
};

// 32-byte global accesses (two adjacent groups), L1 not allocated.  Both
// addresses must be 32-byte aligned.
__device__ __forceinline__ void ld_wide(const char* p, uint4& lo, uint4& hi) {
  uint64_t w0, w1, w2, w3;
  asm volatile("ld.global.L1::no_allocate.v4.b64 {%0,%1,%2,%3}, [%4];"
               : "=l"(w0), "=l"(w1), "=l"(w2), "=l"(w3)
               : "l"(p));
  lo = make_uint4((uint32_t)w0, (uint32_t)(w0 >> 32), (uint32_t)w1, (uint32_t)(w1 >> 32));
  hi = make_uint4((uint32_t)w2, (uint32_t)(w2 >> 32), (uint32_t)w3, (uint32_t)(w3 >> 32));
}

__device__ __forceinline__ void st_wide(char* p, uint4 lo, uint4 hi) {
  const uint64_t w0 = lo.x | ((uint64_t)lo.y << 32), w1 = lo.z | ((uint64_t)lo.w << 32);
  const uint64_t w2 = hi.x | ((uint64_t)hi.y << 32), w3 = hi.z | ((uint64_t)hi.w << 32);
  asm volatile("st.global.L1::no_allocate.v4.b64 [%0], {%1,%2,%3,%4};" ::"l"(p), "l"(w0), "l"(w1),
               "l"(w2), "l"(w3)
               : "memory");
}

// Calls with at least this many 16-byte groups per rank (4 MiB) use 32-byte
// requests where the kernels allow them: measured faster from ~2 Mi bf16
// elements per rank up and slower below (R = 8, GB300).
constexpr size_t kWideMinGroups = (size_t)1 << 18;

__device__ __forceinline__ bool aligned32(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 31u) == 0;
}

// One element's bits (2 or 4 bytes) at p.
template <int kBytes>
__device__ __forceinline__ uint32_t ld_elem(const char* p) {
  if (kBytes == 2) {
    unsigned short v;
    asm volatile("ld.global.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
  } else {
    uint32_t v;
    asm volatile("ld.global.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
  }
}

template <int kBytes>
__device__ __forceinline__ void st_elem(char* p, uint32_t v) {
  if (kBytes == 2) {
    asm volatile("st.global.u16 [%0], %1;" ::"l"(p), "h"((unsigned short)v) : "memory");
  } else {
    asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
  }
}

// Load group g (16 bytes) of a buffer.  `valid` < E::kGroup only for the
// last, partial group; `vec` is false when some pointer of the call is not
// 16-byte aligned.  Missing elements read as zero bits (never stored back).
template <class E, bool kHint = false>
__device__ __forceinline__ uint4 load_group(const char* base, size_t g, int valid, bool vec,
                                            uint64_t pol = 0) {
  const char* p = base + g * kGroupBytes;
  if (vec && valid == E::kGroup) return ld_v4_stream<kHint>(p, pol);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int e = 0; e < E::kGroup; ++e) {
    if (e < valid) {
      const uint32_t bits = ld_elem<E::kBytes>(p + e * E::kBytes);
      constexpr int per_word = 4 / E::kBytes;
      const uint32_t h = bits << (8 * E::kBytes * (e % per_word));
      if (e / per_word == 0) w[0] |= h;
      else if (e / per_word == 1) w[1] |= h;
      else if (e / per_word == 2) w[2] |= h;
      else w[3] |= h;
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <class E, bool kHint = false>
__device__ __forceinline__ void store_group(char* base, size_t g, uint4 v, int valid, bool vec,
                                            uint64_t pol = 0) {
  char* p = base + g * kGroupBytes;
  if (vec && valid == E::kGroup) {
    st_v4_stream<kHint>(p, v, pol);
    return;
  }
#pragma unroll
  for (int e = 0; e < E::kGroup; ++e) {
    if (e < valid) {
      constexpr int per_word = 4 / E::kBytes;
      const int wi = e / per_word;
      const uint32_t w = wi == 0 ? v.x : wi == 1 ? v.y : wi == 2 ? v.z : v.w;
      const uint32_t bits =
          E::kBytes == 4 ? w : (w >> (8 * E::kBytes * (e % per_word))) & 0xFFFFu;
      st_elem<E::kBytes>(p + e * E::kBytes, bits);
    }
  }
}

// Number of valid elements in group g of a buffer of `count` elements.
template <class E>
__device__ __forceinline__ int group_valid(size_t g, size_t count) {
  const size_t first = g * E::kGroup;
  const size_t left = count - first;
  return left >= (size_t)E::kGroup ? E::kGroup : (int)left;
}

// Copy the R input and output pointers of a call into shared memory, and
// decide (CTA-uniformly) whether every pointer allows 16-byte vectors.
template <int R>
__device__ __forceinline__ bool load_tables(const CallArgs& a, const char** s_in, char** s_out) {
  __shared__ int s_misaligned;
  if (threadIdx.x == 0) s_misaligned = 0;
  __syncthreads();
  if (threadIdx.x < R) {
    const char* p = a.in_tbl[threadIdx.x];
    s_in[threadIdx.x] = p;
    if (reinterpret_cast<uintptr_t>(p) & 15u) atomicOr(&s_misaligned, 1);
  } else if (threadIdx.x < 2 * R) {
    char* p = a.out_tbl[threadIdx.x - R];
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
  bool pdl = false;  // launch with programmatic dependent launch (plain kernels only)
};

// Programmatic dependent launch.  A kernel launched with cfg.pdl may be
// scheduled while the previous kernel in its stream is still running; its
// first statement waits until that kernel has completed and its memory
// operations are visible (griddepcontrol.wait), then lets the next kernel
// be scheduled (griddepcontrol.launch_dependents).  No kernel touches global
// memory before that wait, so results are those of plain stream order; what
// is saved is the launch gap between back-to-back calls.  Launched without
// the attribute, both instructions have nothing to wait for or release.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch configuration of a plain (non-cooperative) kernel.
inline cudaLaunchConfig_t plain_config(const LaunchCfg& cfg, dim3 grid, size_t smem,
                                       cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = dim3((unsigned)cfg.threads);
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = cfg.pdl ? 1 : 0;
  return lc;
}

// Launchers (defined in the kernel translation units).  `dtype` is an
// ar_dtype_t; each returns the CUDA error of its launch(es).
cudaError_t launch_oneshot_pull(int R, int dtype, const CallArgs& a, LaunchCfg cfg, cudaStream_t s);
cudaError_t launch_oneshot_fanout(int R, int dtype, const CallArgs& a, LaunchCfg cfg,
                                  cudaStream_t s);
cudaError_t launch_twophase(int R, int dtype, const CallArgs& a, LaunchCfg cfg, cudaStream_t s);
cudaError_t launch_fused_ll8(int R, int dtype, const CallArgs& a, const FusedArgs& f,
                             LaunchCfg cfg, cudaStream_t s);
cudaError_t launch_fused_ll8_staged(int R, int dtype, const CallArgs& a, const FusedArgs& f,
                                    LaunchCfg cfg, cudaStream_t s);
cudaError_t launch_packet_3op(int R, int dtype, const CallArgs& a, const FusedArgs& f,
                              LaunchCfg cfg, cudaStream_t s);
// Reduce-scatter / all-gather (k_rs_ag.cu): a.count is the block length;
// the grid is (cfg.ctas, R).
cudaError_t launch_reduce_scatter(int R, int dtype, const CallArgs& a, LaunchCfg cfg,
                                  cudaStream_t s);
cudaError_t launch_all_gather(int R, int dtype, const CallArgs& a, LaunchCfg cfg, cudaStream_t s);

// Occupancy (CTAs per SM) of the grid-sized kernels for R ranks, dtype and
// `threads` threads per CTA.
int fused_ctas_per_sm(int R, int dtype, int threads);
int fused_staged_ctas_per_sm(int R, int dtype, int threads);
int fanout_ctas_per_sm(int R, int dtype, int threads);

// Bulk-copy fan-out (k_oneshot_bulk.cu): fixed 256 threads per CTA, dynamic
// shared memory per CTA, CTAs per SM, and a one-time attribute set-up.
constexpr int kBulkThreads = 256;
size_t bulk_smem_bytes(int R);
int bulk_ctas_per_sm(int R, int dtype);
cudaError_t bulk_prepare(int R, int dtype);
cudaError_t launch_oneshot_fanout_bulk(int R, int dtype, const CallArgs& a, LaunchCfg cfg,
                                       cudaStream_t s);

// Whether every input group offset (R * shard_groups) and packet slot offset
// (R * R * slot_groups) of a fused call fits in 32 bits.
inline int fused_fits_32bit(int R, size_t shard_groups, size_t slot_groups) {
  const unsigned long long lim = 0xFFFFFFFFull;
  return (unsigned long long)R * shard_groups < lim &&
         (unsigned long long)R * (unsigned long long)R * slot_groups < lim;
}

// The write-mode fused kernel runs one clique per CTA: R warp groups of Tr
// threads each (Tr a multiple of 32), group r standing for virtual rank r.
// Tr for a requested CTA size of `threads`: threads / R rounded down to a
// multiple of 32, at least 32.
inline int fused_rank_threads(int R, int threads) {
  const int tr = threads / R / 32 * 32;
  return tr < 32 ? 32 : tr;
}

// Elements per 16-byte group of an ar_dtype_t (0 for an unknown one).
inline int group_elems(int dtype) {
  return dtype == AR_FP32 ? 4 : (dtype == AR_BF16 || dtype == AR_FP16) ? 8 : 0;
}

}  // namespace ar

// Dispatch on a runtime (R, dtype) to CALL(RR, EE) with RR a compile-time
// rank count and EE an element type, inside a function returning
// cudaError_t (an unsupported pair returns cudaErrorInvalidValue).
#define AR_R_CASE(CALL, EE, RR) \
  case RR:                      \
    CALL(RR, EE);               \
    break;
#define AR_SWITCH_R8(R, CALL, EE)                                                           \
  switch (R) {                                                                            \
    AR_R_CASE(CALL, EE, 1) AR_R_CASE(CALL, EE, 2) AR_R_CASE(CALL, EE, 3)                  \
    AR_R_CASE(CALL, EE, 4) AR_R_CASE(CALL, EE, 5) AR_R_CASE(CALL, EE, 6)                  \
    AR_R_CASE(CALL, EE, 7) AR_R_CASE(CALL, EE, 8)                                         \
    default: return cudaErrorInvalidValue;                                                \
  }
#define AR_SWITCH_R16(R, CALL, EE)                                                          \
  switch (R) {                                                                            \
    AR_R_CASE(CALL, EE, 1) AR_R_CASE(CALL, EE, 2) AR_R_CASE(CALL, EE, 3)                  \
    AR_R_CASE(CALL, EE, 4) AR_R_CASE(CALL, EE, 5) AR_R_CASE(CALL, EE, 6)                  \
    AR_R_CASE(CALL, EE, 7) AR_R_CASE(CALL, EE, 8) AR_R_CASE(CALL, EE, 9)                  \
    AR_R_CASE(CALL, EE, 10) AR_R_CASE(CALL, EE, 11) AR_R_CASE(CALL, EE, 12)               \
    AR_R_CASE(CALL, EE, 13) AR_R_CASE(CALL, EE, 14) AR_R_CASE(CALL, EE, 15)               \
    AR_R_CASE(CALL, EE, 16)                                                               \
    default: return cudaErrorInvalidValue;                                                \
  }
#define AR_DISPATCH(DT, R, CALL, SWITCH)          \
  switch (DT) {                                   \
    case AR_BF16: SWITCH(R, CALL, ::ar::Bf16) break; \
    case AR_FP16: SWITCH(R, CALL, ::ar::F16) break;  \
    case AR_FP32: SWITCH(R, CALL, ::ar::F32) break;  \
    default: return cudaErrorInvalidValue;        \
  }
