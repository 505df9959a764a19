// Reduce-scatter and all-gather over the same R virtual ranks.
//
// "Add HIP-graph capture coverage for the sharded-relay collectives"
// (meta-pytorch/torchcomms #3850) serves reduce-scatter and allreduce with
// one push-reduce kernel that differs only in a per-peer source stride and
// an owner offset (reduce-scatter: stride = recvCount, offset = slot *
// recvCount; allreduce: both 0).  Here the same one-shot read serves both:
//
//   reduce-scatter: rank s's input holds R blocks of `recvcount` elements;
//     out_r[j] = round(sum over s in rank order of in_s[r*recvcount + j]).
//     The CTAs of grid row r (blockIdx.y = r) read block r of all R inputs
//     once and write out_r: (R*R + R)*recvcount elements moved.
//   all-gather: out_r[s*sendcount + j] = in_s[j] for every r; grid row s
//     reads in_s once and writes it into all R outputs (write mode):
//     (R + R*R)*sendcount elements moved.
//
// Vector (16-byte) accesses need every pointer 16-byte aligned and the block
// length a multiple of the group (8 elements of 2 bytes, 4 of fp32) so that
// every block starts aligned; otherwise the call uses element-sized
// accesses.  Outputs must not overlap inputs.
#include "ar_internal.cuh"

namespace ar {
namespace {

template <int R, class E>
__global__ void __launch_bounds__(512) k_reduce_scatter(CallArgs a) {
  __shared__ const char* s_in[R];
  __shared__ char* s_out[R];
  // The caller's pointer tables are read before waiting for the previous
  // kernel in the stream (programmatic dependent launch), so that round trip
  // overlaps its tail; inputs and outputs are touched only after the wait.
  const bool vec = load_tables<R>(a, s_in, s_out) && (a.count % E::kGroup == 0);
  pdl_enter();
  const int r = blockIdx.y;
  const size_t base = (size_t)r * a.count * E::kBytes;  // byte offset of block r
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t j = (size_t)blockIdx.x * blockDim.x + threadIdx.x; j < a.groups; j += stride) {
    const int valid = group_valid<E>(j, a.count);
    uint4 x[R];
#pragma unroll
    for (int s = 0; s < R; ++s) x[s] = load_group<E>(s_in[s] + base, j, valid, vec);
    Acc<E> acc;
    acc.set(x[0]);
#pragma unroll
    for (int s = 1; s < R; ++s) acc.add(x[s]);
    store_group<E>(s_out[r], j, acc.round(), valid, vec);
  }
}

template <int R, class E>
__global__ void __launch_bounds__(512) k_all_gather(CallArgs a) {
  __shared__ const char* s_in[R];
  __shared__ char* s_out[R];
  // The caller's pointer tables are read before waiting for the previous
  // kernel in the stream (programmatic dependent launch), so that round trip
  // overlaps its tail; inputs and outputs are touched only after the wait.
  const bool vec = load_tables<R>(a, s_in, s_out) && (a.count % E::kGroup == 0);
  pdl_enter();
  const int s = blockIdx.y;
  const size_t base = (size_t)s * a.count * E::kBytes;  // byte offset of block s in every output
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t j = (size_t)blockIdx.x * blockDim.x + threadIdx.x; j < a.groups; j += stride) {
    const int valid = group_valid<E>(j, a.count);
    const uint4 x = load_group<E>(s_in[s], j, valid, vec);
#pragma unroll
    for (int r = 0; r < R; ++r) store_group<E>(s_out[r] + base, j, x, valid, vec);
  }
}

}  // namespace

cudaError_t launch_reduce_scatter(int R, int dtype, const CallArgs& a, LaunchCfg cfg,
                                  cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t lc = plain_config(cfg, dim3((unsigned)cfg.ctas, (unsigned)R), 0, s, attr);
#define L(RR, EE) return cudaLaunchKernelEx(&lc, k_reduce_scatter<RR, EE>, a)
  AR_DISPATCH(dtype, R, L, AR_SWITCH_R16)
#undef L
  return cudaErrorInvalidValue;
}

cudaError_t launch_all_gather(int R, int dtype, const CallArgs& a, LaunchCfg cfg, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t lc = plain_config(cfg, dim3((unsigned)cfg.ctas, (unsigned)R), 0, s, attr);
#define L(RR, EE) return cudaLaunchKernelEx(&lc, k_all_gather<RR, EE>, a)
  AR_DISPATCH(dtype, R, L, AR_SWITCH_R16)
#undef L
  return cudaErrorInvalidValue;
}

}  // namespace ar
