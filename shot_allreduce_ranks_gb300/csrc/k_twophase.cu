// Two-phase allreduce: the two-stage scheme of "optimize allreduce write mode
// by broadcast output ptr" (ROCm/aiter #1910) in its original form, before
// write mode.
//
//   launch 1 (stage 1, reduce-scatter): the 16-byte groups are split into R
//     shards of ceil(groups / R); owner o reduces shard o over all R inputs
//     and stores it into its own output out_o only.
//   launch 2 (stage 2, broadcast): owner o reads shard o back from out_o and
//     stores it into every other rank's output.
//
// Stage 2 re-reads the reduced shard from HBM: the "one access to local HBM"
// that the aiter page's write mode removes.  Total traffic 4*R*N + 2*N bytes
// for 2-byte elements (twice that for fp32).
// The kernel boundary orders stage 1's stores before stage 2's loads; it
// also makes in-place calls safe (all inputs are consumed in launch 1).
#include "ar_internal.cuh"

namespace ar {
namespace {

// CTA b works for owner b % R on chunk b / R (gridDim.x is a multiple of R).
template <int R, class E>
__global__ void __launch_bounds__(512) k_twophase_reduce(CallArgs a) {
  __shared__ const char* s_in[R];
  __shared__ char* s_out[R];
  // The caller's pointer tables are read before waiting for the previous
  // kernel in the stream (programmatic dependent launch), so that round trip
  // overlaps its tail; inputs and outputs are touched only after the wait.
  const bool vec = load_tables<R>(a, s_in, s_out);
  pdl_enter();
  const int o = (int)(blockIdx.x % R);
  const size_t g0 = (size_t)o * a.shard_groups;
  if (g0 >= a.groups) return;
  const size_t n = min(a.shard_groups, a.groups - g0);
  const size_t stride = (size_t)(gridDim.x / R) * blockDim.x;
  for (size_t j = (size_t)(blockIdx.x / R) * blockDim.x + threadIdx.x; j < n; j += stride) {
    const size_t g = g0 + j;
    const int valid = group_valid<E>(g, a.count);
    uint4 x[R];
#pragma unroll
    for (int s = 0; s < R; ++s) x[s] = load_group<E>(s_in[s], g, valid, vec);
    Acc<E> acc;
    acc.set(x[0]);
#pragma unroll
    for (int s = 1; s < R; ++s) acc.add(x[s]);
    store_group<E>(s_out[o], g, acc.round(), valid, vec);
  }
}

template <int R, class E>
__global__ void __launch_bounds__(512) k_twophase_broadcast(CallArgs a) {
  __shared__ const char* s_in[R];
  __shared__ char* s_out[R];
  // The caller's pointer tables are read before waiting for the previous
  // kernel in the stream (programmatic dependent launch), so that round trip
  // overlaps its tail; inputs and outputs are touched only after the wait.
  const bool vec = load_tables<R>(a, s_in, s_out);
  pdl_enter();
  const int o = (int)(blockIdx.x % R);
  const size_t g0 = (size_t)o * a.shard_groups;
  if (g0 >= a.groups) return;
  const size_t n = min(a.shard_groups, a.groups - g0);
  const size_t stride = (size_t)(gridDim.x / R) * blockDim.x;
  for (size_t j = (size_t)(blockIdx.x / R) * blockDim.x + threadIdx.x; j < n; j += stride) {
    const size_t g = g0 + j;
    const int valid = group_valid<E>(g, a.count);
    const uint4 y = load_group<E>(s_out[o], g, valid, vec);
#pragma unroll
    for (int s = 0; s < R; ++s)
      if (s != o) store_group<E>(s_out[s], g, y, valid, vec);
  }
}

}  // namespace

cudaError_t launch_twophase(int R, int dtype, const CallArgs& a, LaunchCfg cfg, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t lc = plain_config(cfg, dim3((unsigned)cfg.ctas), 0, s, attr);
  cudaError_t e = cudaErrorInvalidValue;
#define L(RR, EE) e = cudaLaunchKernelEx(&lc, k_twophase_reduce<RR, EE>, a)
  AR_DISPATCH(dtype, R, L, AR_SWITCH_R16)
#undef L
  if (e != cudaSuccess || R == 1) return e;
#define L(RR, EE) e = cudaLaunchKernelEx(&lc, k_twophase_broadcast<RR, EE>, a)
  AR_DISPATCH(dtype, R, L, AR_SWITCH_R16)
#undef L
  return e;
}

}  // namespace ar
