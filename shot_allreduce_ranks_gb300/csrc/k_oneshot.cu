// One-shot allreduce kernels: every element's R inputs are read and summed in
// a single pass, with no intermediate buffer.
//
//  * pull   -- the one-shot allreduce of "One shot all reduce Example"
//              (pytorch-labs/helion #245): the CTA standing for rank r reads
//              the chunk from all R ranks' buffers and writes only out_r.
//              Ranks are the fastest grid dimension, so the R CTAs reading
//              one chunk run together and share its lines in L2.
//  * fanout -- the same read, combined with the write mode of "optimize
//              allreduce write mode by broadcast output ptr" (ROCm/aiter
//              #1910, Motivation): one thread reads a 16-byte group of every
//              rank once, reduces it, and stores the result into all R
//              outputs through the output-pointer table.  4*R*N bytes move
//              for 2-byte elements (8*R*N for fp32), the minimum.  For large
//              calls (at least kWideMinGroups groups, R <= 8, every pointer
//              32-byte aligned) each access moves two adjacent groups as one
//              32-byte request: measured 13.30 vs 13.85 us at 440x5120 and
//              22.6 vs 24.2 us at 512x8192 (R = 8, bf16), but slower below
//              about 2 Mi elements (3.79 vs 3.39 us at 256 Ki), hence the size
//              threshold.
//
// Both handle any count (the last group may be partial) and fall back to
// element-sized accesses for a call whose pointers are not all 16-byte
// aligned.
#include "ar_internal.cuh"

namespace ar {
namespace {

template <int R, class E>
__device__ __forceinline__ uint4 reduce_group(const char* const* s_in, size_t g, int valid,
                                              bool vec) {
  uint4 x[R];
#pragma unroll
  for (int s = 0; s < R; ++s) x[s] = load_group<E>(s_in[s], g, valid, vec);
  Acc<E> acc;
  acc.set(x[0]);
#pragma unroll
  for (int s = 1; s < R; ++s) acc.add(x[s]);
  return acc.round();
}

// Grid-stride over groups, two groups (g, g + stride) per iteration for
// R <= 8 so that 2R independent 16-byte loads are in flight per thread
// before any store; one group per iteration above 8 ranks (registers).
// Fan-out with 32-byte requests: pair p = groups 2p and 2p+1 of every rank;
// the last whole group (if the count of whole groups is odd) and a partial
// group go one group at a time.  Every pointer is 32-byte aligned.
template <int R, class E>
__device__ __forceinline__ void fanout_wide(const CallArgs& a, const char* const* s_in,
                                            char* const* s_out) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t g0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t npairs = (a.count / E::kGroup) / 2;
  for (size_t p = g0; p < npairs; p += stride) {
    uint4 lo[R], hi[R];
#pragma unroll
    for (int s = 0; s < R; ++s) ld_wide(s_in[s] + p * 2 * kGroupBytes, lo[s], hi[s]);
    Acc<E> al, ah;
    al.set(lo[0]);
    ah.set(hi[0]);
#pragma unroll
    for (int s = 1; s < R; ++s) {
      al.add(lo[s]);
      ah.add(hi[s]);
    }
    const uint4 yl = al.round(), yh = ah.round();
#pragma unroll
    for (int r = 0; r < R; ++r) st_wide(s_out[r] + p * 2 * kGroupBytes, yl, yh);
  }
  for (size_t t = 2 * npairs + g0; t < a.groups; t += stride) {
    const int valid = group_valid<E>(t, a.count);
    const uint4 y = reduce_group<R, E>(s_in, t, valid, true);
#pragma unroll
    for (int r = 0; r < R; ++r) store_group<E>(s_out[r], t, y, valid, true);
  }
}

template <int R, class E>
__global__ void __launch_bounds__(512) k_oneshot_fanout(CallArgs a) {
  __shared__ const char* s_in[R];
  __shared__ char* s_out[R];
  // The caller's pointer tables are read before waiting for the previous
  // kernel in the stream (programmatic dependent launch), so that round trip
  // overlaps its tail; inputs and outputs are touched only after the wait.
  const bool vec = load_tables<R>(a, s_in, s_out);
  pdl_enter();
  if constexpr (R <= 8) {
    if (vec && a.groups >= kWideMinGroups) {
      bool all32 = true;
#pragma unroll
      for (int s = 0; s < R; ++s) all32 = all32 && aligned32(s_in[s]) && aligned32(s_out[s]);
      if (all32) {
        fanout_wide<R, E>(a, s_in, s_out);
        return;
      }
    }
  }
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if constexpr (R <= 8) {
    for (; g + stride < a.groups; g += 2 * stride) {
      const size_t g2 = g + stride;
      const int valid2 = group_valid<E>(g2, a.count);
      uint4 x[R], y[R];
#pragma unroll
      for (int s = 0; s < R; ++s) {
        x[s] = load_group<E>(s_in[s], g, E::kGroup, vec);
        y[s] = load_group<E>(s_in[s], g2, valid2, vec);
      }
      Acc<E> ax, ay;
      ax.set(x[0]);
      ay.set(y[0]);
#pragma unroll
      for (int s = 1; s < R; ++s) {
        ax.add(x[s]);
        ay.add(y[s]);
      }
      const uint4 rx = ax.round(), ry = ay.round();
#pragma unroll
      for (int r = 0; r < R; ++r) {
        store_group<E>(s_out[r], g, rx, E::kGroup, vec);
        store_group<E>(s_out[r], g2, ry, valid2, vec);
      }
    }
  }
  for (; g < a.groups; g += stride) {
    const int valid = group_valid<E>(g, a.count);
    const uint4 y = reduce_group<R, E>(s_in, g, valid, vec);
#pragma unroll
    for (int r = 0; r < R; ++r) store_group<E>(s_out[r], g, y, valid, vec);
  }
}

// gridDim.x is a multiple of R; CTA b stands for rank b % R and chunk b / R.
// If some output pointer equals some input pointer (in-place use), a CTA
// writing out_r could overwrite data another rank's CTA has yet to read, so
// the kernel detects that case on the device and lets the rank-0 CTA of each
// chunk write every output instead (the fan-out order, alias-safe).
template <int R, class E>
__global__ void __launch_bounds__(512) k_oneshot_pull(CallArgs a) {
  __shared__ const char* s_in[R];
  __shared__ char* s_out[R];
  __shared__ int s_alias;
  // The caller's pointer tables are read before waiting for the previous
  // kernel in the stream (programmatic dependent launch), so that round trip
  // overlaps its tail; inputs and outputs are touched only after the wait.
  const bool vec = load_tables<R>(a, s_in, s_out);
  pdl_enter();
  if (threadIdx.x == 0) {
    int alias = 0;
    for (int r = 0; r < R; ++r)
      for (int s = 0; s < R; ++s) alias |= (s_out[r] == s_in[s]);
    s_alias = alias;
  }
  __syncthreads();
  const bool alias = s_alias != 0;
  const int r = (int)(blockIdx.x % R);
  if (alias && r != 0) return;
  const size_t chunks = gridDim.x / R;
  const size_t stride = chunks * blockDim.x;
  for (size_t g = (size_t)(blockIdx.x / R) * blockDim.x + threadIdx.x; g < a.groups; g += stride) {
    const int valid = group_valid<E>(g, a.count);
    const uint4 y = reduce_group<R, E>(s_in, g, valid, vec);
    if (alias) {
#pragma unroll
      for (int q = 0; q < R; ++q) store_group<E>(s_out[q], g, y, valid, vec);
    } else {
      store_group<E>(s_out[r], g, y, valid, vec);
    }
  }
}

}  // namespace

static cudaError_t fanout_occ(int R, int dtype, int threads, int* n) {
#define Q(RR, EE) \
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, k_oneshot_fanout<RR, EE>, threads, 0)
  AR_DISPATCH(dtype, R, Q, AR_SWITCH_R16)
#undef Q
  return cudaErrorInvalidValue;
}

int fanout_ctas_per_sm(int R, int dtype, int threads) {
  int n = 0;
  return fanout_occ(R, dtype, threads, &n) == cudaSuccess ? n : 0;
}

cudaError_t launch_oneshot_fanout(int R, int dtype, const CallArgs& a, LaunchCfg cfg,
                                  cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t lc = plain_config(cfg, dim3((unsigned)cfg.ctas), 0, s, attr);
#define L(RR, EE) return cudaLaunchKernelEx(&lc, k_oneshot_fanout<RR, EE>, a)
  AR_DISPATCH(dtype, R, L, AR_SWITCH_R16)
#undef L
  return cudaErrorInvalidValue;
}

cudaError_t launch_oneshot_pull(int R, int dtype, const CallArgs& a, LaunchCfg cfg,
                                cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t lc = plain_config(cfg, dim3((unsigned)cfg.ctas), 0, s, attr);
#define L(RR, EE) return cudaLaunchKernelEx(&lc, k_oneshot_pull<RR, EE>, a)
  AR_DISPATCH(dtype, R, L, AR_SWITCH_R16)
#undef L
  return cudaErrorInvalidValue;
}

}  // namespace ar
