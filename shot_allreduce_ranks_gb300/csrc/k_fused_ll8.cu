// Fused LL8 packet allreduce: the write-mode kernel and its comparison forms.
//
// This is the monolithic fused packet allreduce of "Add monolithic fused
// packet allreduce kernel and Model::all_reduce_packet API" (microsoft/ark
// #254, Changes): scatter -> reduce -> broadcast in one kernel, synchronised
// by low-latency (LL) packet flags instead of cross-block barriers.  The R
// virtual ranks live on one GPU, so "remote" scratch is a region of this
// GPU's memory, and the threads standing for a rank touch only what that
// rank's GPU would touch: its own input, the packet slots it owns or sends
// to, and (write mode) every rank's output.
//
// The 16-byte groups are split into R shards of ceil(groups / R); rank o
// owns shard o.
//   scatter (packet stores): rank r reads group j of every other owner o's
//     shard from its own input and stores it, as four LL8 packets, into
//     owner o's slot for source r.
//   reduce (packet polls): owner r loads, for every other source s, the four
//     packets of group j from its slot for s until all four carry the
//     expected flag, takes its own input for position r, and sums the R
//     contributions in rank order 0..R-1 in fp32.
//   broadcast (write mode): owner r rounds once and stores the group into
//     all R outputs through the output-pointer table, as in "optimize
//     allreduce write mode by broadcast output ptr" (ROCm/aiter #1910,
//     Motivation); completion is the kernel boundary, so no packets flow
//     back.
//
// k_fused_ll8 runs the three steps pipelined over rounds, with one clique
// of R warp groups per CTA (its comment below).  Its write-mode instance is
// AR_FUSED_LL8; the instance without write mode (AR_FUSED_LL8_STAGED) sends
// the result back as packets, the ARK page's own form, so the two differ in
// that step alone.  The three-launch decomposition (AR_PACKET_3OP) runs each
// phase over the whole message with a CTA per virtual rank (b % R), one
// kernel per phase.
//
// LL8 packet: one 64-bit word, low 32 bits = one 32-bit word of a group (two
// bf16/fp16, lower-indexed element in the low half, or one fp32), high 32
// bits = flag.  Stores and loads are 64-bit strong (relaxed, gpu scope)
// accesses, four packets per 32-byte vector instruction; the memory model
// treats each 64-bit element as single-copy atomic, so a packet whose flag
// matches carries that call's data.
//
// Flag rotation.  The ARK page leaves Flag = 1 hardcoded (Known limitations);
// here the flag is a device-resident epoch in [1, 2^32-1] that skips 0 (the
// value of zeroed scratch).  Because the epoch never comes from the host, a
// CUDA-graph replay rotates it too (the by-value epoch hazard G2 of "Add
// HIP-graph capture coverage for the sharded-relay collectives",
// meta-pytorch/torchcomms #3850), and it never rewinds while the handle
// lives (that page's region-lifetime commit).  A packet left from an earlier
// call carries an older flag, so it reads as not yet arrived.
//
// Every wait is bounded: after the spin limit the thread records a timeout
// in the device error word and abandons the call; other waiters see the
// abandoned epoch and stop too.
#include <string.h>

#include <algorithm>
#include <mutex>

#include "ar_internal.cuh"

namespace ar {
namespace {

constexpr int kFusedMaxThreads = 512;
// The write-mode kernel for R <= 4 is compiled for at most 256 threads and
// three CTAs per SM (80 registers instead of 128, a third clique per SM).
// Against the 128-register build (R = 4, bf16, graph replay) it is faster
// from about 2 Mi elements per rank up (10.7 vs 11.3 us at 2.2 Mi, 18.3 vs
// 19.7 at 4 Mi, 63.3 vs 68.5 at 16 Mi, 133.7 vs 138.5 at 32 Mi; R = 3 at
// 4 Mi 14.3 vs 19.2) and slower below, where a CTA has one or two tiles
// (4.8 vs 4.2 us at 512 Ki, 7.4 vs 6.7 at 1 Mi, with any grid; the one-shot
// kernels serve those sizes).  The form without write mode keeps the wider
// bound: at 80 registers its receive spills and it was 9-20% slower.  Host
// code finds the limit through fused_ctas_per_sm (zero CTAs per SM above
// it).
template <int R, bool kWriteMode>
constexpr int fused_bound_threads() { return kWriteMode && R <= 4 ? 256 : kFusedMaxThreads; }
template <int R, bool kWriteMode>
constexpr int fused_bound_ctas() { return kWriteMode && R <= 4 ? 3 : 1; }
constexpr uint32_t kMaxSpins = 1u << 24;

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// The pipelined fused kernel treats DevState's epoch (low word) and done
// (high word) as one 64-bit location.  Every DevState sits at a 256-byte
// boundary (cudaMalloc, or the allocation-free path's __align__(256) array).
static_assert(offsetof(DevState, epoch) % 8 == 0 &&
                  offsetof(DevState, done) == offsetof(DevState, epoch) + 4,
              "epoch and done must form one aligned 64-bit word, epoch first");
__device__ __forceinline__ uint64_t* epoch_done(DevState* st) {
  return reinterpret_cast<uint64_t*>(&st->epoch);
}

__device__ __forceinline__ uint64_t atom_add_relaxed_u64(uint64_t* p, uint64_t v) {
  uint64_t old;
  asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Four packets of one group in one 32-byte access, flag in the high half of
// every 64-bit word.  Stores ask L2 to keep the line (it is read back soon by
// the owner); loads mark it evict-first once read.  As a vector access, the
// memory model treats it as four 64-bit accesses, each single-copy atomic.
// kCta: strong at CTA scope only, which suffices when the producer and the
// owner are threads of one CTA (the pipelined kernel's cliques).  The
// write-mode instance uses it (R = 8, bf16, same-call A/B against GPU scope:
// 38.2 vs 38.4 us at 512x8192, 135.0 vs 137.8 at 16 Mi elements, 261.2 vs
// 268.3 at 32 Mi; R = 6: 233.0 vs 236.2 at 32 Mi); the instance without
// write mode keeps GPU scope, which was faster for it (R = 6: 337 vs 366 us,
// R = 4: 215 vs 222 at 32 Mi), as does the three-launch form, whose
// producers and owners are in different CTAs.
template <bool kCta = false>
__device__ __forceinline__ void st_packets(uint64_t* p, uint4 x, uint32_t epoch) {
  const uint64_t hi = (uint64_t)epoch << 32;
  if (kCta)
    asm volatile("st.relaxed.cta.global.L2::evict_last.v4.b64 [%0], {%1,%2,%3,%4};" ::"l"(p),
                 "l"(hi | x.x), "l"(hi | x.y), "l"(hi | x.z), "l"(hi | x.w)
                 : "memory");
  else
    asm volatile("st.relaxed.gpu.global.L2::evict_last.v4.b64 [%0], {%1,%2,%3,%4};" ::"l"(p),
                 "l"(hi | x.x), "l"(hi | x.y), "l"(hi | x.z), "l"(hi | x.w)
                 : "memory");
}

struct Packets4 {
  uint64_t w[4];
  template <bool kCta = false>
  __device__ __forceinline__ void load(const uint64_t* p) {
    if (kCta)
      asm volatile("ld.relaxed.cta.global.L2::evict_first.v4.b64 {%0,%1,%2,%3}, [%4];"
                   : "=l"(w[0]), "=l"(w[1]), "=l"(w[2]), "=l"(w[3])
                   : "l"(p));
    else
      asm volatile("ld.relaxed.gpu.global.L2::evict_first.v4.b64 {%0,%1,%2,%3}, [%4];"
                   : "=l"(w[0]), "=l"(w[1]), "=l"(w[2]), "=l"(w[3])
                   : "l"(p));
  }
  __device__ __forceinline__ bool arrived(uint32_t epoch) const {
    return (uint32_t)(w[0] >> 32) == epoch && (uint32_t)(w[1] >> 32) == epoch &&
           (uint32_t)(w[2] >> 32) == epoch && (uint32_t)(w[3] >> 32) == epoch;
  }
  __device__ __forceinline__ uint4 data() const {
    return make_uint4((uint32_t)w[0], (uint32_t)w[1], (uint32_t)w[2], (uint32_t)w[3]);
  }
};

// Packet slot (a, b != a) of a region laid out [a][b packed, skipping a]
// [group][4]: for scatter packets a = owner, b = source; for result packets
// (the staged variants) a = destination rank, b = owner.
template <int R>
__device__ __forceinline__ uint64_t* slot_ptr(uint64_t* region, size_t slot_groups, int a, int b) {
  const int slot = a * (R - 1) + (b < a ? b : b - 1);
  return region + (size_t)slot * slot_groups * 4;
}

// Records the first timeout in the (sticky) error word and marks this
// call's epoch as abandoned, so the call's other waiters stop early while
// later calls, which carry newer epochs, are unaffected.
__device__ __noinline__ void report_timeout(const FusedArgs& f, int owner, uint32_t pending,
                                            uint32_t epoch) {
  const int missing = __ffs((int)pending) - 1;
  if (atomicCAS(&f.state->error, kDevErrNone, kDevErrTimeout) == kDevErrNone)
    f.state->error_info = ((uint32_t)owner << 16) | (uint32_t)missing;
  atomicAdd(&f.state->timeouts, 1u);
  st_relaxed_u32(&f.state->abort_epoch, epoch);
}

// Per-thread view of one launch of a three-launch-form kernel.
struct Lane {
  int r;              // virtual rank this CTA stands for (blockIdx.x % R)
  size_t t0, tstride; // first group and group stride of this thread within a shard
  size_t Vs;          // groups per shard
  uint32_t epoch;
  bool vec;
  uint64_t pol_in;    // evict-first policy for input reads
};

template <int R>
__device__ __forceinline__ Lane make_lane(const CallArgs& a, uint32_t epoch, bool vec) {
  Lane l;
  l.r = (int)(blockIdx.x % R);
  l.t0 = (size_t)(blockIdx.x / R) * blockDim.x + threadIdx.x;
  l.tstride = (size_t)(gridDim.x / R) * blockDim.x;
  l.Vs = a.shard_groups;
  l.epoch = epoch;
  l.vec = vec;
  l.pol_in = l2_policy_evict_first();
  return l;
}

// Prologue of every packet kernel: pointer tables into shared memory, the
// call's epoch read once by thread 0 and shared with the CTA.
template <int R>
__device__ __forceinline__ Lane packet_prologue(const CallArgs& a, const FusedArgs& f,
                                                const char** s_in, char** s_out) {
  __shared__ uint32_t s_epoch;
  const bool vec = load_tables<R>(a, s_in, s_out);
  if (threadIdx.x == 0) s_epoch = ld_relaxed_u32(&f.state->epoch);
  __syncthreads();
  return make_lane<R>(a, s_epoch, vec);
}

// Waits until every packet set s in `pending` (already loaded once into
// pk[s]) carries `flag`, re-polling ptr(s).  Bounded: after spin_limit_ns of
// %globaltimer (or an iteration cap, a backstop in case the timer did not
// advance; every iteration is at least one L2 round trip) it records a
// timeout and returns false; it also returns false as soon as another
// waiter of the same call (identified by its base epoch) has given up.
// Entry i stands for position base + i in the list of sources; with
// skip >= 0 that list holds only the other ranks (position p is source
// p < skip ? p : p + 1), otherwise position s is source s.  limit_mul
// stretches the limits for waits on packets that are sent only after their
// sender's own wait succeeded (result packets), so that when a producer is
// missing, a wait on its own packets runs out first and is the one reported.
template <int N, bool kCta = false, class Ptr>
__device__ __forceinline__ bool wait_packets_at(const FusedArgs& f, Packets4 (&pk)[N],
                                                uint32_t pending, uint32_t flag,
                                                uint32_t call_epoch, int who, Ptr ptr,
                                                int skip = -1, int base = 0,
                                                uint32_t limit_mul = 1) {
#pragma unroll
  for (int s = 0; s < N; ++s)
    if ((pending & (1u << s)) && pk[s].arrived(flag)) pending &= ~(1u << s);
  if (!pending) return true;
  uint64_t t_first = 0;
  uint32_t spins = 0;
  while (pending) {
    __nanosleep(32);
#pragma unroll
    for (int s = 0; s < N; ++s) {
      if (pending & (1u << s)) {
        pk[s].template load<kCta>(ptr(s));
        if (pk[s].arrived(flag)) pending &= ~(1u << s);
      }
    }
    if (pending && (++spins & 15u) == 0) {
      const uint64_t now = global_timer_ns();
      if (spins == 16u) t_first = now;
      if (spins / limit_mul > kMaxSpins ||
          (spins > 16u && now - t_first > f.spin_limit_ns * limit_mul)) {
        pending <<= base;
        if (skip >= 0)
          pending = (pending & ((1u << skip) - 1u)) | ((pending >> skip) << (skip + 1));
        report_timeout(f, who, pending, call_epoch);
        return false;
      }
      if (ld_relaxed_u32(&f.state->abort_epoch) == call_epoch) return false;
    }
  }
  return true;
}

// The same wait on a region laid out like the scatter scratch.
template <int R>
__device__ __forceinline__ bool wait_packets(const FusedArgs& f, uint64_t* region, int a_idx,
                                             size_t j, Packets4 (&pk)[R], uint32_t pending,
                                             uint32_t epoch) {
  return wait_packets_at<R>(f, pk, pending, epoch, epoch, a_idx, [&](int s) {
    return slot_ptr<R>(region, f.slot_groups, a_idx, s) + j * 4;
  });
}

// ---- scatter: rank r's slices of every other owner's shard, as packets ----
// Two groups (j, j + tstride) per iteration: all 2(R-1) loads are issued
// before the first packet store.
template <int R, class E>
__device__ __forceinline__ void phase_scatter(const CallArgs& a, const FusedArgs& f, const Lane& l,
                                              const char* my_in) {
  if constexpr (R == 1) return;
  if (l.r == f.skip_producer) return;
  for (size_t j = l.t0; j < l.Vs; j += 2 * l.tstride) {
    const size_t j2 = j + l.tstride;
    uint4 x[R > 1 ? R - 1 : 1], y[R > 1 ? R - 1 : 1];
#pragma unroll
    for (int k = 1; k < R; ++k) {
      const int o = (l.r + k) % R;
      const size_t g = (size_t)o * l.Vs + j;
      if (g < a.groups)
        x[k - 1] = load_group<E, true>(my_in, g, group_valid<E>(g, a.count), l.vec, l.pol_in);
      const size_t g2 = (size_t)o * l.Vs + j2;
      if (j2 < l.Vs && g2 < a.groups)
        y[k - 1] = load_group<E, true>(my_in, g2, group_valid<E>(g2, a.count), l.vec, l.pol_in);
    }
#pragma unroll
    for (int k = 1; k < R; ++k) {
      const int o = (l.r + k) % R;
      uint64_t* slot = slot_ptr<R>(f.scratch, f.slot_groups, o, l.r);
      const size_t g = (size_t)o * l.Vs + j;
      if (g < a.groups) st_packets(slot + j * 4, x[k - 1], l.epoch);
      const size_t g2 = (size_t)o * l.Vs + j2;
      if (j2 < l.Vs && g2 < a.groups) st_packets(slot + j2 * 4, y[k - 1], l.epoch);
    }
  }
}

// ---- reduce owner r's shard ------------------------------------------------
// Polls the R-1 sources' packets of each group, sums the R contributions in
// rank order (own input at position r), rounds once.  kWriteMode: store the
// group into all R outputs.  Otherwise: store it into out_r only and send it
// as result packets to every other rank's result slot for owner r.
// Returns false if the call was abandoned after a timeout.
template <int R, class E, bool kWriteMode>
__device__ __forceinline__ bool phase_reduce(const CallArgs& a, const FusedArgs& f, const Lane& l,
                                             const char* my_in, char* const* s_out) {
  const size_t g0 = (size_t)l.r * l.Vs;
  const size_t n = g0 < a.groups ? min(l.Vs, a.groups - g0) : 0;
  for (size_t j = l.t0; j < n; j += l.tstride) {
    const size_t g = g0 + j;
    const int valid = group_valid<E>(g, a.count);
    const uint4 own = load_group<E, true>(my_in, g, valid, l.vec, l.pol_in);
    Packets4 pk[R];
    uint32_t pending = 0;
#pragma unroll
    for (int s = 0; s < R; ++s)
      if (s != l.r) {
        pk[s].load(slot_ptr<R>(f.scratch, f.slot_groups, l.r, s) + j * 4);
        pending |= 1u << s;
      }
    const bool ok = wait_packets<R>(f, f.scratch, l.r, j, pk, pending, l.epoch);
    if (!ok) return false;
    Acc<E> acc;
    acc.set(l.r == 0 ? own : pk[0].data());
#pragma unroll
    for (int s = 1; s < R; ++s) acc.add(s == l.r ? own : pk[s].data());
    const uint4 y = acc.round();
    if (kWriteMode) {
#pragma unroll
      for (int q = 0; q < R; ++q) store_group<E>(s_out[q], g, y, valid, l.vec);
    } else {
      store_group<E>(s_out[l.r], g, y, valid, l.vec);
#pragma unroll
      for (int q = 0; q < R; ++q)
        if (q != l.r) st_packets(slot_ptr<R>(f.rscratch, f.slot_groups, q, l.r) + j * 4, y, l.epoch);
    }
  }
  return true;
}

// ---- receive: rank r copies every other owner's reduced shard out of its
// result slots into out_r (the three-launch form's last step) ----------------
template <int R, class E>
__device__ __forceinline__ bool phase_recv(const CallArgs& a, const FusedArgs& f, const Lane& l,
                                           char* const* s_out) {
  if constexpr (R == 1) return true;
  char* my_out = s_out[l.r];
  for (size_t j = l.t0; j < l.Vs; j += l.tstride) {
    Packets4 pk[R];
    uint32_t pending = 0;
#pragma unroll
    for (int o = 0; o < R; ++o)
      if (o != l.r && (size_t)o * l.Vs + j < a.groups) {
        pk[o].load(slot_ptr<R>(f.rscratch, f.slot_groups, l.r, o) + j * 4);
        pending |= 1u << o;
      }
    const uint32_t present = pending;
    if (!wait_packets<R>(f, f.rscratch, l.r, j, pk, pending, l.epoch)) return false;
#pragma unroll
    for (int o = 0; o < R; ++o)
      if (present & (1u << o)) {
        const size_t g = (size_t)o * l.Vs + j;
        store_group<E>(my_out, g, pk[o].data(), group_valid<E>(g, a.count), l.vec);
      }
  }
  return true;
}

// ---- flag rotation: the last CTA of the call's last kernel advances the
// epoch (skipping 0) and resets the done counter ------------------------------
__device__ __forceinline__ void epoch_advance_to(const FusedArgs& f, uint32_t next) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(&f.state->done, 1u);
    if (prev == gridDim.x - 1) {
      __threadfence();
      st_relaxed_u32(&f.state->done, 0u);
      st_relaxed_u32(&f.state->epoch, next);
    }
  }
}

// The epoch sequence skips 0 (the value of zeroed scratch): the k-th value
// after e.
__device__ __forceinline__ uint32_t flag_at(uint32_t e, uint64_t k) {
  return (uint32_t)(((uint64_t)e - 1u + k) % 0xFFFFFFFFull + 1u);
}

__device__ __forceinline__ void epoch_advance(const FusedArgs& f, uint32_t epoch) {
  epoch_advance_to(f, flag_at(epoch, 1));
}

// Drops one 128-byte line from L2 without writing it back; its memory
// contents keep whatever was last written back (an older packet or zeros).
__device__ __forceinline__ void discard_l2_line(const uint64_t* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// After every lane of a warp has read its packets of the tile starting at
// group jt: drop the warp's lines (4 groups of 32 bytes each, 8 lines per
// source for 32 lanes) that hold some group < n of owner r's slots.
template <int R>
__device__ __forceinline__ void discard_round(const uint64_t* region, size_t slot_groups, int r,
                                              size_t jt, size_t t, size_t n) {
  const size_t wb = jt + (t & ~(size_t)31);  // the warp's first group
  for (int i = (int)(t & 31); i < 8 * (R - 1); i += 32) {
    const size_t line_g = wb + (size_t)(i & 7) * 4;
    if (line_g < n)
      discard_l2_line(region + ((size_t)(r * (R - 1) + (i >> 3)) * slot_groups + line_g) * 4);
  }
}

// Test hook: a bounded wait of `ns` of %globaltimer (a late producer).
__device__ __noinline__ void producer_delay(uint64_t ns) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0; i < kMaxSpins && global_timer_ns() - t0 < ns; ++i) __nanosleep(256);
}

// Scatter -> reduce -> broadcast, pipelined over tiles.  kWriteMode: the
// owner stores the sum straight into all R outputs.  Without it (the ARK
// page's form) the owner stores its own output and sends the sum to every
// other rank as result packets (a second packet region, same slot layout
// with a = destination); rank r receives round k - 2 lead in its iteration
// k, one lead after the owners reduced it, and copies the R - 1 shards into
// out_r.
//
// A CTA is a clique: R warp groups of Tr threads (Tr a multiple of 32), group
// r standing for virtual rank r, so producers and owners that exchange
// packets always sit on the same SM and no CTA ever waits on another.  A
// tile is Tr consecutive groups of every shard (one group per thread); CTA c
// works on tiles c, c + C, c + 2C, ... (its rounds).  Iteration k of a warp
// group scatters its rank's slices of round k (one group per other owner
// per thread) and reduces its own shard's group of round k - lead, whose
// packets the clique stored `lead` iterations earlier, so polls mostly
// succeed at once.  The input slices of round k + 1 are loaded right after
// round k's packet stores (when their registers are free), so their latency
// overlaps the reduce.
//
// Packets written but not yet read stay within about lead + 1 rounds of the
// grid (R(R-1) * 32 bytes per tile group), a few tens of MB, so they live in
// L2 whatever the message size.  With f.discard, after a warp has read its
// 32 groups of a round (eight 128-byte lines per source) it drops those
// lines from L2, so consumed packets are never written back to HBM.  In ring
// mode (f.ring_rounds = D > 0, for large messages) the packets of round k go
// instead to slot k mod D of a ring private to the CTA, at the thread's
// index, and carry the round's own flag (epoch + k; the call moves the epoch
// on by its rounds); a CTA barrier at the end of every iteration lets a slot
// be reused only once every warp of the CTA has read it (D = lead + 1), so
// the lines are overwritten while still in L2 and never written back.
//
// Two bodies: iterations whose tiles lie wholly inside every shard (whole
// 16-byte groups, aligned buffers, offsets within 32 bits: nearly all of
// them) run without per-group checks; the others (the ragged end of the
// message, misaligned buffers) take the checked body.  Whole tiles come
// first, so each body is a loop of its own.  Both use the same packet layout
// and produce the same bits.
//
// Deadlock freedom: iteration i of a warp waits only on warps of its own CTA:
// on scatters of round i - lead, done in their iteration i - lead; without
// write mode, on result packets of round i - 2 lead, sent in their iteration
// i - lead; in ring mode, on the barrier every warp of the CTA reaches at the
// end of each iteration.  By induction on i every wait is eventually
// satisfied.  The waits are bounded all the same.
template <int R, class E, bool kWriteMode = true>
__global__ void __launch_bounds__(fused_bound_threads<R, kWriteMode>(),
                                  fused_bound_ctas<R, kWriteMode>()) k_fused_ll8(CallArgs a, FusedArgs f) {
  constexpr int RO = R > 1 ? R - 1 : 1;  // entries for the other ranks
  __shared__ const char* s_in[R];
  __shared__ char* s_out[R];
  __shared__ uint32_t s_epoch;
  __shared__ int s_misaligned;
  // Launched with programmatic dependent launch.  The caller's pointer
  // tables are read first, overlapping the previous kernel's tail; then the
  // kernel waits until that kernel has completed and its writes (the epoch
  // among them) are visible, and lets the next one be scheduled, before it
  // reads the epoch or touches any input, output or packet.  Flag rotation at
  // arrival: thread 2R reads the epoch and counts its CTA in with one 64-bit
  // atomic on {epoch, done}; the CTA whose count completes the grid writes
  // {next epoch, 0} in one 64-bit store at its end, so no CTA waits on
  // another at exit.  Every access this kernel makes to the pair is to that
  // one location, so coherence alone orders each CTA's read (its atomic, all
  // of them before the last one) before that store; no fence is needed.  The
  // next call, ordered after this kernel, reads the new epoch.
  uint32_t arrival = 0;
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
  // CTA c is clique c; its warp group r (Tr threads, a multiple of 32)
  // stands for virtual rank r.
  const size_t Tr = blockDim.x / R;
  const int r = (int)(threadIdx.x / Tr);
  const size_t t = threadIdx.x % Tr;
  const size_t C = gridDim.x, c = blockIdx.x;
  const size_t Vs = a.shard_groups;
  const uint64_t pol_in = l2_policy_evict_first();
  const size_t g0 = (size_t)r * Vs;  // first group of my shard
  const size_t my_n = g0 < a.groups ? min(Vs, a.groups - g0) : 0;
  const size_t my_n_max = min(Vs, a.groups);  // positions any shard's packets may use
  const size_t tiles = (Vs + Tr - 1) / Tr;
  const size_t K = c < tiles ? (tiles - c + C - 1) / C : 0;  // rounds of this clique
  const size_t L = (size_t)(f.lead > 0 ? f.lead : 1);
  // Iterations after the last scatter: the reduce trails by L, and without
  // write mode the receive of the result packets trails the reduce by L.
  const size_t LL = kWriteMode ? L : 2 * L;
  const bool scatter_on = R > 1 && r != f.skip_producer;

  const uint32_t Vs32 = (uint32_t)Vs, SG32 = (uint32_t)f.slot_groups;
  // Per-rank offsets for q = 1..R-1 (owner o = (r + q) % R), in shared memory
  // to leave the registers to the data in flight: start of o's shard in
  // rank r's input, and start of the slot (owner o, source r).
  __shared__ uint32_t s_in_off[R][RO], s_dst_off[R][RO];
  // Ring mode: packets of round k live in slot k % D of this CTA's ring,
  // at the thread's index instead of its shard position, and carry the flag
  // of their round (the call moves the epoch on by its rounds).
  const bool ring = kWriteMode && f.ring_rounds > 0;
  const uint32_t D = ring ? (uint32_t)f.ring_rounds : 1u;
  const uint32_t Tr32 = (uint32_t)Tr, t32 = (uint32_t)t;
  const uint32_t sstride = ring ? Tr32 : SG32;  // groups per (owner, source) slot
  const uint32_t RRT = (uint32_t)(R * (R - 1)) * Tr32;  // groups per ring round of a CTA
  const uint32_t ring_cta = (uint32_t)c * D * RRT;
  uint64_t* const pkt = ring ? f.ring : f.scratch;
  if (t > 0 && t < (size_t)R) {
    const int q = (int)t, o = r + q < R ? r + q : r + q - R;
    s_in_off[r][q - 1] = (uint32_t)o * Vs32;
    s_dst_off[r][q - 1] = (uint32_t)(o * (R - 1) + (r < o ? r : r - 1)) * sstride;
  }
  __syncthreads();  // tables and offsets visible; all of this overlapped the previous kernel
  pdl_enter();
  if (threadIdx.x == 2 * R) {
    const uint64_t old = atom_add_relaxed_u64(epoch_done(f.state), 1ull << 32);
    s_epoch = (uint32_t)old;
    arrival = (uint32_t)(old >> 32);
  }
  const bool vec = s_misaligned == 0;
  // Fast body: tiles [jt, jt + Tr) with jt + Tr <= fast_vs are whole groups
  // in every shard (the last shard is the shortest).
  const size_t whole = a.count / E::kGroup;
  const size_t fast_vs =
      (vec && f.fast32 && whole > (size_t)(R - 1) * Vs) ? min(Vs, whole - (size_t)(R - 1) * Vs)
                                                        : 0;
  const char* my_in = s_in[r];
  // The input slices of round k are loaded during iteration k - 1, right
  // after that iteration's packet stores (when their registers are free), so
  // their HBM latency overlaps the reduce of iteration k - 1.  Round 0's are
  // issued here, before the epoch's round trip completes.
  uint4 x[RO];
  auto load_slices = [&](size_t kk) {
    const uint32_t js = (uint32_t)((c + kk * C) * Tr + t);
#pragma unroll
    for (int q = 0; q < R - 1; ++q)
      x[q] = ld_v4_stream<true>(my_in + (size_t)(s_in_off[r][q] + js) * kGroupBytes, pol_in);
  };
  {
    const size_t nf0 = fast_vs / Tr;
    const bool whole0 = nf0 > c;  // round 0 of this clique is a whole tile
    if (scatter_on && whole0 && K > 0) load_slices(0);
  }
  __syncthreads();  // the epoch
  const uint32_t epoch = s_epoch;
  // Slot of (owner r, i-th other source in rank order): r * (R - 1) + i.
  const uint32_t src_row = (uint32_t)(r * (R - 1)) * sstride;
  const uint32_t own_off = (uint32_t)r * Vs32;
  // Position of this thread's packets of round kk within a slot: its shard
  // position, or (ring mode) its index in the round's slot of the ring.
  auto ppos = [&](size_t kk, uint32_t jpos) -> uint32_t {
    return ring ? ring_cta + (uint32_t)(kk % D) * RRT + t32 : jpos;
  };
  auto flag_of = [&](size_t kk) -> uint32_t { return ring ? flag_at(epoch, kk) : epoch; };
  // Rounds of the call: the epoch moves on by this many flags (ring mode).
  const size_t K_all = (tiles + C - 1) / C;
  // Iterations whose tiles are all whole form a prefix [0, k_fast): tile
  // c + kC is whole for k < kf (the same for every warp of the CTA).
  const size_t nf = fast_vs / Tr;
  const size_t kf = nf > c ? (nf - c + C - 1) / C : 0;
  const size_t k_fast = kf >= K ? K + LL : kf;
  // End of an iteration: in ring mode a CTA barrier (a ring slot is reused
  // only after every warp of the CTA has read it; all threads leave the loop
  // together), else a warp vote.
  auto iteration_done = [&](bool good) -> bool {
    return ring ? __syncthreads_and(good) != 0 : __all_sync(0xFFFFFFFFu, good);
  };

  if (r == f.delay_rank && f.delay_ns) producer_delay(f.delay_ns);

  bool ok = true;
  size_t k = 0;
  for (; k < k_fast; ++k) {
    // ---------------- whole tiles: 32-bit offsets, no per-group checks
    const size_t jts = (c + k * C) * Tr;                       // scatter tile (round k)
    const bool rd_round = k >= L && k < K + L;
    const size_t jtr = rd_round ? (c + (k - L) * C) * Tr : 0;  // reduced tile (round k - L)
    {
      const bool sc = scatter_on && k < K;
      const uint32_t js = (uint32_t)(jts + t), jr = (uint32_t)(jtr + t);
      const uint32_t pr = rd_round ? ppos(k - L, jr) : 0u;
      Packets4 pk[RO];
      uint4 own = make_uint4(0, 0, 0, 0);
      if (rd_round) {
        own = ld_v4_stream<true>(my_in + (size_t)(own_off + jr) * kGroupBytes, pol_in);
#pragma unroll
        for (int i = 0; i < R - 1; ++i)
          pk[i].load<kWriteMode>(pkt + (size_t)(src_row + (uint32_t)i * sstride + pr) * 4);
      }
      if (sc) {
        const uint32_t ps = ppos(k, js), fl = flag_of(k);
#pragma unroll
        for (int q = 0; q < R - 1; ++q)
          st_packets<kWriteMode>(pkt + (size_t)(s_dst_off[r][q] + ps) * 4, x[q], fl);
      }
      const bool preload = scatter_on && k + 1 < K && k + 1 < k_fast;
      if (kWriteMode && preload) load_slices(k + 1);
      if (rd_round) {
        ok = wait_packets_at<RO, kWriteMode>(
            f, pk, R > 1 ? (1u << (R - 1)) - 1u : 0u, flag_of(k - L), epoch, r,
            [&](int i) { return pkt + (size_t)(src_row + (uint32_t)i * sstride + pr) * 4; }, r);
        if (ok) {
          // rank order 0..R-1; entry i of pk is source i (< r) or i + 1 (> r)
          Acc2<E> acc;
#pragma unroll
          for (int s = 0; s < R; ++s) {
            uint4 v = own;
            if (s < R - 1 && s < r) v = pk[s < R - 1 ? s : 0].data();
            else if (s > 0 && s > r) v = pk[s > 0 ? s - 1 : 0].data();
            if (s == 0) acc.set(v);
            else acc.add(v);
          }
          const uint4 y = acc.round();
          const size_t goff = (size_t)(own_off + jr) * kGroupBytes;
          if (kWriteMode) {
#pragma unroll
            for (int q = 0; q < R; ++q) st_v4_stream(s_out[q] + goff, y);
          } else {
            // own output, and the sum as result packets to every other rank
            st_v4_stream(s_out[r] + goff, y);
#pragma unroll
            for (int q = 0; q < R - 1; ++q)
              st_packets<kWriteMode>(f.rscratch + (size_t)(s_dst_off[r][q] + jr) * 4, y, epoch);
          }
        }
      }
      // Without write mode: receive the result packets of round k - 2L from
      // every other owner and copy them into this rank's output, at most four
      // owners at a time; the next round's slices are loaded once the first
      // chunk's loads are out (the reduce's registers are free by then).
      if (!kWriteMode) {
        constexpr int kChunk = RO < 4 ? RO : 4;
        const bool rv = R > 1 && k >= 2 * L;
        const uint32_t jq = rv ? (uint32_t)((c + (k - 2 * L) * C) * Tr + t) : 0u;
        const uint64_t* const rrow = f.rscratch + (size_t)(src_row + jq) * 4;
#pragma unroll
        for (int i0 = 0; i0 < RO; i0 += kChunk) {
          constexpr int kN = kChunk;
          const int n = RO - i0 < kN ? RO - i0 : kN;
          Packets4 rk[kN];
          if (rv) {
#pragma unroll
            for (int i = 0; i < kN; ++i)
              if (i < n) rk[i].load<kWriteMode>(rrow + (size_t)(i0 + i) * sstride * 4);
          }
          if (i0 == 0 && preload) load_slices(k + 1);
          if (rv && R > 1) {
            ok = ok && wait_packets_at<kN, kWriteMode>(
                           f, rk, (1u << n) - 1u, epoch, epoch, r,
                           [&](int i) { return rrow + (size_t)(i0 + i) * sstride * 4; }, r, i0,
                           2u);
            if (ok) {
#pragma unroll
              for (int i = 0; i < kN; ++i)
                if (i < n) {
                  const uint32_t o = (uint32_t)(i0 + i < r ? i0 + i : i0 + i + 1);
                  st_v4_stream(s_out[r] + (size_t)(o * Vs32 + jq) * kGroupBytes, rk[i].data());
                }
            }
          }
        }
      }
    }
    if (!iteration_done(ok)) {
      ok = false;
      break;
    }
    if (R > 1 && f.discard && !ring) {
      if (rd_round) discard_round<R>(f.scratch, f.slot_groups, r, jtr, t, my_n);
      if (!kWriteMode && k >= 2 * L)
        discard_round<R>(f.rscratch, f.slot_groups, r, (c + (k - 2 * L) * C) * Tr, t, my_n_max);
    }
  }
  for (; ok && k < K + LL; ++k) {
    // ---------------- checked body (ragged end, misaligned buffers)
    const size_t jts = (c + k * C) * Tr;
    const bool rd_round = k >= L && k < K + L;
    const size_t jtr = rd_round ? (c + (k - L) * C) * Tr : 0;
    {
      const size_t js = jts + t;
      const bool sc = scatter_on && k < K && js < Vs;
      uint4 x[RO];
      if (sc) {
#pragma unroll
        for (int q = 1; q < R; ++q) {
          const size_t g = (size_t)((r + q) % R) * Vs + js;
          if (g < a.groups)
            x[q - 1] = load_group<E, true>(my_in, g, group_valid<E>(g, a.count), vec, pol_in);
        }
      }
      const size_t jr = jtr + t;
      const bool rd = rd_round && jr < my_n;
      Packets4 pk[R];
      uint4 own = make_uint4(0, 0, 0, 0);
      uint32_t pending = 0;
      if (rd) {
        own = load_group<E, true>(my_in, g0 + jr, group_valid<E>(g0 + jr, a.count), vec,
                                  pol_in);
#pragma unroll
        for (int s = 0; s < R; ++s)
          if (s != r) {
            pk[s].load<kWriteMode>(slot_ptr<R>(pkt, sstride, r, s) + (size_t)ppos(k - L, (uint32_t)jr) * 4);
            pending |= 1u << s;
          }
      }
      if (sc) {
#pragma unroll
        for (int q = 1; q < R; ++q) {
          const int o = (r + q) % R;
          if ((size_t)o * Vs + js < a.groups)
            st_packets<kWriteMode>(slot_ptr<R>(pkt, sstride, o, r) + (size_t)ppos(k, (uint32_t)js) * 4,
                       x[q - 1], flag_of(k));
        }
      }
      if (rd) {
        const size_t pr = ppos(k - L, (uint32_t)jr);
        ok = wait_packets_at<R, kWriteMode>(f, pk, pending, flag_of(k - L), epoch, r, [&](int s) {
          return slot_ptr<R>(pkt, sstride, r, s) + pr * 4;
        });
        if (ok) {
          Acc2<E> acc;
          acc.set(r == 0 ? own : pk[0].data());
#pragma unroll
          for (int s = 1; s < R; ++s) acc.add(s == r ? own : pk[s].data());
          const uint4 y = acc.round();
          const size_t g = g0 + jr;
          const int valid = group_valid<E>(g, a.count);
          if (kWriteMode) {
#pragma unroll
            for (int q = 0; q < R; ++q) store_group<E>(s_out[q], g, y, valid, vec);
          } else {
            store_group<E>(s_out[r], g, y, valid, vec);
#pragma unroll
            for (int q = 1; q < R; ++q)
              st_packets<kWriteMode>(slot_ptr<R>(f.rscratch, f.slot_groups, (r + q) % R, r) + jr * 4, y, epoch);
          }
        }
      }
      // Receive (ragged end): one owner at a time.
      if (!kWriteMode && R > 1 && k >= 2 * L) {
        const size_t jq = (c + (k - 2 * L) * C) * Tr + t;
        for (int o = 0; ok && o < R; ++o) {
          const size_t g = (size_t)o * Vs + jq;
          if (o == r || jq >= Vs || g >= a.groups) continue;
          const uint64_t* const p = slot_ptr<R>(f.rscratch, f.slot_groups, r, o) + jq * 4;
          Packets4 rk[1];
          rk[0].load<kWriteMode>(p);
          ok = wait_packets_at<1, kWriteMode>(f, rk, 1u, epoch, epoch, r, [&](int) { return p; }, -1, o,
                                              2u);
          if (ok) store_group<E>(s_out[r], g, rk[0].data(), group_valid<E>(g, a.count), vec);
        }
      }
    }
    if (!iteration_done(ok)) {
      ok = false;
      break;
    }
    if (R > 1 && f.discard && !ring) {
      if (rd_round) discard_round<R>(f.scratch, f.slot_groups, r, jtr, t, my_n);
      if (!kWriteMode && k >= 2 * L)
        discard_round<R>(f.rscratch, f.slot_groups, r, (c + (k - 2 * L) * C) * Tr, t, my_n_max);
    }
  }
  if (threadIdx.x == 2 * R && arrival == gridDim.x - 1)
    st_relaxed_u64(epoch_done(f.state), (uint64_t)flag_at(epoch, ring ? K_all : 1));
}

// The three-launch decomposition the ARK page replaced (send_packet ->
// recv_reduce_send_packet -> recv_packet): the same phases, one kernel each,
// ordered by kernel boundaries instead of by co-residency.
template <int R, class E>
__global__ void __launch_bounds__(kFusedMaxThreads) k_packet_send(CallArgs a, FusedArgs f) {
  __shared__ const char* s_in[R];
  __shared__ char* s_out[R];
  const Lane l = packet_prologue<R>(a, f, s_in, s_out);
  phase_scatter<R, E>(a, f, l, s_in[l.r]);
}

template <int R, class E>
__global__ void __launch_bounds__(kFusedMaxThreads) k_packet_reduce_send(CallArgs a, FusedArgs f) {
  __shared__ const char* s_in[R];
  __shared__ char* s_out[R];
  const Lane l = packet_prologue<R>(a, f, s_in, s_out);
  phase_reduce<R, E, false>(a, f, l, s_in[l.r], s_out);
}

template <int R, class E>
__global__ void __launch_bounds__(kFusedMaxThreads) k_packet_recv(CallArgs a, FusedArgs f) {
  __shared__ const char* s_in[R];
  __shared__ char* s_out[R];
  const Lane l = packet_prologue<R>(a, f, s_in, s_out);
  phase_recv<R, E>(a, f, l, s_out);
  epoch_advance(f, l.epoch);
}

}  // namespace

namespace {

// CTAs per SM of `threads` threads; zero above the kernel's launch bound,
// which the occupancy query alone does not report.
template <class Kernel>
cudaError_t occ_within_bound(Kernel kernel, int threads, int* n) {
  cudaFuncAttributes fa;
  const cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  if (threads > fa.maxThreadsPerBlock) {
    *n = 0;
    return cudaSuccess;
  }
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, kernel, threads, 0);
}

cudaError_t occ_fused(int R, int dtype, int threads, int* n) {
#define Q(RR, EE) return occ_within_bound(k_fused_ll8<RR, EE>, threads, n)
  AR_DISPATCH(dtype, R, Q, AR_SWITCH_R8)
#undef Q
  return cudaErrorInvalidValue;
}

cudaError_t occ_staged(int R, int dtype, int threads, int* n) {
#define Q(RR, EE) return occ_within_bound(k_fused_ll8<RR, EE, false>, threads, n)
  AR_DISPATCH(dtype, R, Q, AR_SWITCH_R8)
#undef Q
  return cudaErrorInvalidValue;
}

}  // namespace

int fused_ctas_per_sm(int R, int dtype, int threads) {
  int n = 0;
  return occ_fused(R, dtype, threads, &n) == cudaSuccess ? n : 0;
}

int fused_staged_ctas_per_sm(int R, int dtype, int threads) {
  int n = 0;
  return occ_staged(R, dtype, threads, &n) == cudaSuccess ? n : 0;
}

cudaError_t launch_fused_ll8(int R, int dtype, const CallArgs& a, const FusedArgs& f,
                             LaunchCfg cfg, cudaStream_t s) {
  // A plain launch: every packet wait stays inside one CTA, so co-residency
  // is not needed for progress (the grid is still sized to fit at once).
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t lc = plain_config(cfg, dim3((unsigned)cfg.ctas), 0, s, attr);
#define L(RR, EE) return cudaLaunchKernelEx(&lc, k_fused_ll8<RR, EE>, a, f)
  AR_DISPATCH(dtype, R, L, AR_SWITCH_R8)
#undef L
  return cudaErrorInvalidValue;
}

cudaError_t launch_fused_ll8_staged(int R, int dtype, const CallArgs& a, const FusedArgs& f,
                                    LaunchCfg cfg, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t lc = plain_config(cfg, dim3((unsigned)cfg.ctas), 0, s, attr);
#define L(RR, EE) return cudaLaunchKernelEx(&lc, k_fused_ll8<RR, EE, false>, a, f)
  AR_DISPATCH(dtype, R, L, AR_SWITCH_R8)
#undef L
  return cudaErrorInvalidValue;
}

cudaError_t launch_packet_3op(int R, int dtype, const CallArgs& a, const FusedArgs& f,
                              LaunchCfg cfg, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
#define L(RR, EE)                                                       \
  k_packet_send<RR, EE><<<cfg.ctas, cfg.threads, 0, s>>>(a, f);         \
  if ((e = cudaGetLastError()) != cudaSuccess) return e;                \
  k_packet_reduce_send<RR, EE><<<cfg.ctas, cfg.threads, 0, s>>>(a, f);  \
  if ((e = cudaGetLastError()) != cudaSuccess) return e;                \
  k_packet_recv<RR, EE><<<cfg.ctas, cfg.threads, 0, s>>>(a, f);         \
  return cudaGetLastError()
  AR_DISPATCH(dtype, R, L, AR_SWITCH_R8)
#undef L
  return cudaErrorInvalidValue;
}

}  // namespace ar

// ---------------------------------------------------------------------------
// Allocation-free entry point: the same fused kernel, with its packet
// scratch and its epoch/counter/error block in fixed device arrays that the
// library image carries, instead of memory a handle allocates.  Every GPU
// that loads this library holds these arrays (AR_NOALLOC_SCRATCH_BYTES plus
// 64 bytes) until the process exits.

namespace {

constexpr size_t kNoAllocWords = AR_NOALLOC_SCRATCH_BYTES / sizeof(uint64_t);
static __device__ __align__(256) uint64_t g_noalloc_scratch[kNoAllocWords];
static __device__ __align__(256) ar::DevState g_noalloc_state;

constexpr int kNoAllocMaxDevices = 64;
constexpr int kNoAllocThreads = 256;

struct NoAllocDevice {
  bool ready;
  uint64_t* scratch;     // device address of g_noalloc_scratch on this device
  ar::DevState* state;   // device address of g_noalloc_state on this device
  int sms;
  int ctas_per_sm[AR_MAX_PACKET_RANKS + 1];
};

NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

// Once per device, with that device current: look up the arrays' device
// addresses (in host code their names are host-side stand-ins, not device
// addresses), zero the scratch so no stale word can carry a live flag, and
// start the epoch at 1.  Synchronous; allocates nothing.
ar_status_t noalloc_setup(int dev, int R, NoAllocDevice* out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    void* scratch = nullptr;
    void* state = nullptr;
    if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess) return AR_ERR_CUDA;
    if (cudaGetSymbolAddress(&state, g_noalloc_state) != cudaSuccess) return AR_ERR_CUDA;
    ar::DevState init;
    memset(&init, 0, sizeof init);
    init.epoch = 1;
    int sms = 0;
    if (cudaMemset(scratch, 0, AR_NOALLOC_SCRATCH_BYTES) != cudaSuccess ||
        cudaMemcpy(state, &init, sizeof init, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return AR_ERR_CUDA;
    d.scratch = static_cast<uint64_t*>(scratch);
    d.state = static_cast<ar::DevState*>(state);
    d.sms = sms;
    d.ready = true;
  }
  if (d.ctas_per_sm[R] == 0)
    d.ctas_per_sm[R] =
        ar::fused_ctas_per_sm(R, AR_BF16, R * ar::fused_rank_threads(R, kNoAllocThreads));
  *out = d;
  return AR_OK;
}

}  // namespace

extern "C" ar_status_t ar_allreduce_fused_noalloc(int R, const void* const* d_in_tbl,
                                                  void* const* d_out_tbl, size_t count,
                                                  void* stream) {
  if (R < 1 || R > AR_MAX_PACKET_RANKS || !d_in_tbl || !d_out_tbl) return AR_ERR_INVALID_ARG;
  if (count == 0) return AR_OK;
  if (count > AR_NOALLOC_MAX_COUNT(R)) return AR_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return AR_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return AR_ERR_UNSUPPORTED;
  NoAllocDevice d;
  ar_status_t st = noalloc_setup(dev, R, &d);
  if (st != AR_OK) return st;
  if (d.ctas_per_sm[R] <= 0) return AR_ERR_CUDA;

  ar::CallArgs a;
  a.in_tbl = reinterpret_cast<const char* const*>(d_in_tbl);
  a.out_tbl = reinterpret_cast<char* const*>(d_out_tbl);
  a.count = count;
  a.groups = (count + 7) / 8;  // bf16: 8 elements per 16-byte group
  a.shard_groups = (a.groups + (size_t)R - 1) / (size_t)R;
  a.state = d.state;
  a.spin_limit_ns = 100ull * 1000ull * 1000ull;
  ar::FusedArgs f;
  f.scratch = d.scratch;
  f.rscratch = nullptr;
  f.slot_groups = a.shard_groups;  // R*(R-1)*slot_groups*32 <= scratch bytes by the check above
  f.state = d.state;
  f.spin_limit_ns = 100ull * 1000ull * 1000ull;
  f.skip_producer = -1;
  // No discards: nothing guarantees that the fixed array's zeros have reached
  // memory, so a dropped line could read back as whatever preceded them.
  f.lead = 1;
  f.discard = 0;
  f.fast32 = ar::fused_fits_32bit(R, a.shard_groups, f.slot_groups);
  f.ring = nullptr;
  f.ring_rounds = 0;
  f.delay_rank = -1;
  f.delay_ns = 0;
  // One clique of R warp groups per CTA, a persistent grid of co-resident CTAs.
  const int tr = ar::fused_rank_threads(R, kNoAllocThreads);
  const size_t limit = (size_t)d.ctas_per_sm[R] * (size_t)d.sms;
  size_t ctas = (a.shard_groups + (size_t)tr - 1) / (size_t)tr;
  ctas = std::max<size_t>(1, std::min(ctas, limit));
  ar::LaunchCfg cfg = {(int)ctas, R * tr};
  return ar::launch_fused_ll8(R, AR_BF16, a, f, cfg, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? AR_OK
             : AR_ERR_CUDA;
}
