// C ABI of the virtual-rank allreduce: handle lifetime, argument checks, the
// per-size variant selector and kernel launches.  Declarations and the
// contract of every entry point are in include/ar.h.
#include <errno.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#include <algorithm>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "ar_internal.cuh"

using ar::CallArgs;
using ar::DevState;
using ar::FusedArgs;
using ar::LaunchCfg;

// ---------------------------------------------------------------------------
// Selector table.  A row applies to calls with count <= max_count for its R
// (R = 0 matches any R); the first matching row wins.  ctas / threads of 0
// mean "use the variant's automatic launch shape".  The built-in rows are
// the crossovers measured on GB300 (one-shot variants below, fan-out above),
// placed where the measured curves meet, as the crossover commit of "Add
// HIP-graph capture coverage for the sharded-relay collectives"
// (meta-pytorch/torchcomms #3850) prescribes, and with the launch shape
// chosen per size instead of one hardcoded block size ("One shot all reduce
// Example", pytorch-labs/helion #245: "performance drop at 1m due to
// hardcoded block_size").
struct TuneRow {
  int R;
  size_t max_count;
  int variant;
  int ctas;
  int threads;
};

// Measured on GB300 (CUDA-graph replay, inputs larger than L2 between
// reuses): one-shot pull is fastest for small messages and fan-out with
// 128-thread CTAs above.  For bf16 the curves cross near 115 Ki elements per
// rank at R = 8 (pull 3.03 us vs 3.28 at 64 Ki; 3.52 vs 3.36 at 128 Ki) and
// near 230 Ki at R = 4 (2.58 vs 2.67 at 128 Ki; 2.83 vs 2.75 at 256 Ki):
// pull reads R^2 N bytes through L2, so the crossover scales as 1/R.  It is
// a number of bytes per rank: fp16 crosses where bf16 does, fp32 at half
// the element count (R = 8: pull 2.91 vs 2.99 us at 32 Ki; 3.36 vs 3.10 at
// 64 Ki), about 1.75 MiB / R per rank.  At R = 16 (bf16) the bulk-copy
// fan-out beats the register fan-out from 64 Ki to 256 Ki elements (3.75 vs
// 4.32 us, 4.16 vs 4.84, 5.11 vs 5.56) and not above (9.26 vs 8.52 at
// 512 Ki, 14.81 vs 13.41 at 1 Mi), hence its end near the geometric mean of
// 256 Ki and 512 Ki (360 Ki elements).  Rows are generated per (R, element
// size) from these rules.
constexpr size_t kPullCrossoverBytesTimesR = 917504 * 2;
constexpr size_t kBulkMaxBytesR16 = 368640 * 2;

std::vector<TuneRow> builtin_table(int R, size_t elem_bytes) {
  const size_t pull_max = kPullCrossoverBytesTimesR / elem_bytes / (size_t)R / 64 * 64;
  std::vector<TuneRow> t = {{R, pull_max, AR_ONESHOT_PULL, 0, 256}};
  if (R >= 16) t.push_back({R, kBulkMaxBytesR16 / elem_bytes, AR_ONESHOT_FANOUT_BULK, 0, 0});
  t.push_back({R, (size_t)-1, AR_ONESHOT_FANOUT, 0, 128});
  return t;
}

struct ar_ctx {
  int R = 0;
  int dtype = AR_BF16;
  size_t elem_bytes = 2;
  size_t max_count = 0;
  int device = 0;
  int num_sms = 0;
  int variant = AR_AUTO;
  LaunchCfg override_cfg[AR_NUM_VARIANTS] = {};
  std::vector<TuneRow> table;
  bool log = false;

  DevState* state = nullptr;
  uint64_t* scratch = nullptr;   // scatter packets
  uint64_t* rscratch = nullptr;  // result packets (staged variants)
  // Allocations behind the packet regions (scratch, rscratch, ring), each
  // with a guard zone before and after the region (guarded_alloc).
  void* region_base[3] = {nullptr, nullptr, nullptr};
  size_t region_bytes[3] = {0, 0, 0};
  size_t scratch_bytes = 0;      // bytes of each region
  size_t slot_groups = 0;
  uint64_t spin_limit_ns = 100ull * 1000ull * 1000ull;
  int skip_producer = -1;
  // The device error block as ar_get_device_status last found it set (it
  // clears the device copy), for ar_last_timeout.
  uint32_t last_error = 0, last_error_info = 0, last_timeouts = 0;
  int delay_rank = -1;         // skewed-producer test hook (persists until cleared)
  uint64_t delay_ns = 0;
  // Packet handling of the write-mode fused kernel, chosen per call from the
  // bytes of packets P = 32 R (R-1) groups-per-shard (measured on GB300,
  // graph replay): P <= L2/2: packets written into the message-sized
  // scratch stay in L2 between calls, so they are left there (R = 8: 22.8 vs
  // 23.5 us at 440x5120 with drops, where packets, inputs and outputs come
  // to 135 MB); L2/2 < P <= 2 L2, or P plus the 4RN bytes of inputs and
  // outputs above 1.1 L2: the scratch, with each consumed line dropped from
  // L2 (R = 8: 38.5 vs 45.6 us at 512x8192 without drops; 67 MB of packets
  // at R = 3, 8 Mi elements: 25.3 vs 30.7 us, and at R = 2, 16 Mi: 35.7 vs
  // 39.9, with 168 and 201 MB in all); P > 2 L2: per-CTA rings of lead + 1
  // rounds with lead 1 (R = 8: 86.8 vs 88.2 us at 10 Mi elements, 103.1 vs
  // 105.4 at 12 Mi, 138.7 vs 145.5 at 16 Mi; R = 4: 90.9 vs 97.9 at 24 Mi,
  // 119.9 vs 134.2 at 32 Mi; below 2 L2 the two were within 3% either way at
  // R = 3 and 4, and the scratch won by 8% at R = 2, 32-48 Mi).  Without
  // write mode (AR_FUSED_LL8_STAGED) the result packets double P, there are
  // no rings, and the lead is 1 (69.1 vs 72.5 us at 512x8192, 530 vs 621 us
  // at 32 Mi elements, 7.0 vs 7.5 us at 4 Ki).  The AR_FUSED_RING,
  // AR_FUSED_DISCARD and AR_FUSED_LEAD environment variables force a choice.
  int fused_lead = 0;          // tiles scattered ahead of the reduce (0: automatic)
  int fused_discard = -1;      // -1 automatic, 0 never, 1 always (scratch mode)
  int l2_bytes = 0;
  bool fused_pdl = true;       // programmatic dependent launch for the pipelined fused kernels
  int fused_ring = -1;         // -1 automatic, 0 never, 1 always
  uint64_t* ring = nullptr;    // the rings of all CTAs
  size_t ring_groups = 0;      // its size in 32-byte packet groups
  int fused_threads = 256;
  int fused_ctas_per_sm = 0;   // occupancy at fused_threads
  // Occupancy cache (CTAs per SM) indexed by threads / 32; 0 = not queried.
  int occ_fused[33] = {};
  int occ_staged[33] = {};
  int occ_fanout[33] = {};
  int bulk_ctas_per_sm = 0;    // bulk fan-out (fixed 256 threads)
  // Programmatic dependent launch for the one-shot, two-phase, reduce-scatter
  // and all-gather kernels of calls that move at most pdl_max_bytes (the
  // pipelined fused kernels: every call; AR_PDL=0: never).  Measured at
  // R = 8, bf16, back-to-back graph-replayed calls: pull 2.34 vs 2.52 us at
  // 4 Ki elements, 2.78 vs 3.15 at 64 Ki; fan-out 3.39 vs 3.77 at 256 Ki;
  // but two-phase 11.2 vs 9.7 us at 1 Mi (32 MiB moved), hence 16 MiB; and
  // two-phase at R = 16 was slower with it already at 16 MiB (11.1 vs 7.1 us
  // at 256 Ki) while faster at R = 8 up to 8 MiB, hence 8 MiB for it.
  bool pdl = true;
  size_t pdl_max_bytes = (size_t)16 << 20;
  size_t pdl_max_bytes_twophase = (size_t)8 << 20;

  // host-buffer path
  char* staging = nullptr;        // 2 * R buffers of max_count elements
  char** staging_tables = nullptr;  // device: R input pointers, then R output pointers
  char** direct_tables = nullptr;   // device: the caller's buffers, when device-accessible
};

namespace {

ar_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? AR_OK : AR_ERR_CUDA; }

// An NVTX range around the host side of one call (what a profiler's timeline
// shows as the call's enqueue).  Without a tool attached it costs a check.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

const char* range_name(int variant) {
  switch (variant) {
    case AR_ONESHOT_PULL: return "ar oneshot_pull";
    case AR_ONESHOT_FANOUT: return "ar oneshot_fanout";
    case AR_TWOPHASE: return "ar twophase";
    case AR_FUSED_LL8: return "ar fused_ll8";
    case AR_ONESHOT_FANOUT_BULK: return "ar oneshot_fanout_bulk";
    case AR_FUSED_LL8_STAGED: return "ar fused_ll8_staged";
    case AR_PACKET_3OP: return "ar packet_3op";
    default: return "ar ?";
  }
}

bool is_packet_variant(int v) {
  return v == AR_FUSED_LL8 || v == AR_FUSED_LL8_STAGED || v == AR_PACKET_3OP;
}

size_t ceil_div(size_t a, size_t b) { return (a + b - 1) / b; }

int parse_variant(const char* s) {
  if (!s || !*s) return -1;
  for (int v = 0; v < AR_NUM_VARIANTS; ++v)
    if (strcmp(s, ar_variant_name(v)) == 0) return v;
  char* end = nullptr;
  long v = strtol(s, &end, 10);
  if (end && *end == '\0' && v >= 0 && v < AR_NUM_VARIANTS) return (int)v;
  return -1;
}

// Table file: one row per line, "R max_count variant [ctas threads]",
// '#' starts a comment; variant by name or number.
bool load_table_file(const char* path, std::vector<TuneRow>* rows) {
  FILE* fp = fopen(path, "r");
  if (!fp) return false;
  char line[512];
  std::vector<TuneRow> out;
  while (fgets(line, sizeof line, fp)) {
    char* hash = strchr(line, '#');
    if (hash) *hash = '\0';
    int R = 0, ctas = 0, threads = 0;
    unsigned long long maxc = 0;
    char vname[64] = {0};
    int n = sscanf(line, "%d %llu %63s %d %d", &R, &maxc, vname, &ctas, &threads);
    if (n <= 0) continue;
    if (n < 3) {
      fclose(fp);
      return false;
    }
    int v = parse_variant(vname);
    if (v <= AR_AUTO) {
      fclose(fp);
      return false;
    }
    out.push_back({R, (size_t)maxc, v, n >= 4 ? ctas : 0, n >= 5 ? threads : 0});
  }
  fclose(fp);
  *rows = out;
  return true;
}

const TuneRow* lookup(const ar_ctx* h, size_t count) {
  for (const TuneRow& t : h->table)
    if ((t.R == 0 || t.R == h->R) && count <= t.max_count) return &t;
  return nullptr;
}

int choose(const ar_ctx* h, size_t count, const TuneRow** row) {
  *row = nullptr;
  if (h->variant != AR_AUTO) return h->variant;
  const TuneRow* t = lookup(h, count);
  *row = t;
  return t ? t->variant : AR_ONESHOT_FANOUT;
}

int occupancy(ar_ctx* h, int variant, int threads) {
  int* cache = variant == AR_FUSED_LL8          ? h->occ_fused
               : variant == AR_FUSED_LL8_STAGED ? h->occ_staged
                                                : h->occ_fanout;
  const int k = threads / 32;
  if (k < 0 || k > 32) return 0;
  if (cache[k] == 0) {
    const int R = h->R, dt = h->dtype;
    const int n = variant == AR_FUSED_LL8          ? ar::fused_ctas_per_sm(R, dt, threads)
                  : variant == AR_FUSED_LL8_STAGED ? ar::fused_staged_ctas_per_sm(R, dt, threads)
                                                   : ar::fanout_ctas_per_sm(R, dt, threads);
    cache[k] = n > 0 ? n : -1;
  }
  return cache[k] > 0 ? cache[k] : 0;
}

// Threads per rank of a fused launch: the request split over R warp groups,
// narrowed while the kernel cannot start a CTA of that size (the write-mode
// kernel for R <= 4 is compiled for at most 256 threads).
int fused_tr(ar_ctx* h, int variant, int threads) {
  int tr = ar::fused_rank_threads(h->R, threads);
  while (tr > 32 && occupancy(h, variant, h->R * tr) == 0) tr -= 32;
  return tr;
}

constexpr int kMaxRingRounds = 3;  // rings are sized for lead 2 (lead + 1 rounds)

// 32-byte packet groups one CTA's ring needs: `rounds` rounds of R(R-1)
// slots of Tr groups.
size_t ring_groups_per_cta(int R, int rounds, int tr) {
  return (size_t)rounds * (size_t)R * (size_t)(R - 1) * (size_t)tr;
}

struct FusedMode {
  int lead;         // tiles scattered ahead of the reduce
  int discard;      // drop consumed scratch lines from L2
  int ring_rounds;  // > 0: per-CTA rings of this many rounds instead of the scratch
};

// The pipelined fused kernel's packet handling for a call with
// `shard_groups` groups per shard and warp groups of `tr` threads (the rules
// at ar_ctx::fused_lead).  Rings only in write mode and where at least one
// CTA's ring fits.  Without write mode the result packets double the
// footprint that decides on the drops.
FusedMode fused_mode(const ar_ctx* h, size_t shard_groups, int tr, bool write_mode) {
  const double P =
      (write_mode ? 1.0 : 2.0) * 32.0 * h->R * (h->R - 1) * (double)shard_groups;
  const double l2 = h->l2_bytes > 0 ? (double)h->l2_bytes : 128.0 * (1 << 20);
  const int ring_lead = h->fused_lead > 0 ? h->fused_lead : 1;
  const bool ring = write_mode && h->ring &&
                    h->ring_groups >= ring_groups_per_cta(h->R, ring_lead + 1, tr) &&
                    (h->fused_ring == 1 || (h->fused_ring < 0 && P > 2.0 * l2));
  FusedMode m;
  m.lead = h->fused_lead > 0 ? h->fused_lead : (ring || !write_mode ? 1 : 2);
  m.ring_rounds = ring ? m.lead + 1 : 0;
  // Write mode also drops the lines when packets, inputs and outputs
  // together (P + 4RN bytes; 32 R^2 bytes per shard group for the last two)
  // overflow L2.
  const double io = 32.0 * h->R * h->R * (double)shard_groups;
  const bool drop = P > 0.5 * l2 || (write_mode && P + io > 1.1 * l2);
  m.discard = ring ? 0 : h->fused_discard >= 0 ? h->fused_discard : (drop ? 1 : 0);
  return m;
}

// Launch shape of one call.  Fan-out: 128 threads, the co-resident grid,
// grown for large calls (its comment); pull and two-phase: 256 threads, one
// group per thread, capped at 16 CTAs per SM, a multiple of R; pipelined
// fused: cliques of R warp groups, min(tiles per shard, co-resident CTAs).
LaunchCfg shape(ar_ctx* h, int variant, const TuneRow* row, size_t groups, size_t shard_groups,
                bool host_memory = false) {
  LaunchCfg c = {0, 0};
  if (row && row->variant == variant) c = {row->ctas, row->threads};
  const LaunchCfg& o = h->override_cfg[variant];
  if (o.ctas > 0) c.ctas = o.ctas;
  if (o.threads > 0) c.threads = o.threads;
  const int R = h->R;
  const size_t cap = (size_t)h->num_sms * 16;
  switch (variant) {
    case AR_ONESHOT_FANOUT: {
      // The co-resident grid (two groups per thread per pass), replaced for
      // large calls by a grid that gives a thread at most G groups: 4 (two
      // 32-byte pairs) for R <= 8, 2 (one pass) above.  A persistent grid
      // looping over a large message was slower (R = 8, bf16, graph replay:
      // 22.4 vs 23.3 us at 512x8192, 41.5 vs 45.1 at 8 Mi elements, 79.4 vs
      // 87.3 at 16 Mi, 155.2 vs 170.9 at 32 Mi; R = 4 at 32 Mi 79.1 vs 88.4;
      // R = 16 at 4 Mi 42.7 vs 45.6), but a grid of up to about 1.5 waves of
      // co-resident CTAs leaves a thin second wave running alone (19.1 vs
      // 18.3 us at 3.2 Mi, 20.0 vs 19.3 at 3.4 Mi), hence the switch at 1.5
      // waves (512x8192 is 1.7).  On page-locked host buffers (the host
      // path) the co-resident grid stays: more CTAs in flight over the host
      // link were slower (553 vs 492 us with 2048 CTAs at 512x8192, 325 vs
      // 290 with 1024 at 440x5120).
      if (c.threads <= 0) c.threads = 128;
      if (c.ctas <= 0) {
        const size_t resident =
            std::max<size_t>(1, (size_t)occupancy(h, variant, c.threads) * (size_t)h->num_sms);
        const size_t T = (size_t)c.threads, G = R <= 8 ? 4 : 2;
        const size_t grown = ceil_div(groups, G * T);
        const bool waves = !host_memory && grown >= resident + resident / 2;
        c.ctas = (int)std::max<size_t>(
            1, waves ? grown : std::min(ceil_div(groups, 2 * T), resident));
      }
      break;
    }
    case AR_ONESHOT_PULL:
    case AR_TWOPHASE: {
      if (c.threads <= 0) c.threads = 256;
      const size_t span = variant == AR_ONESHOT_PULL ? groups : shard_groups;
      if (c.ctas <= 0) {
        const size_t chunks = std::max<size_t>(1, std::min(ceil_div(span, (size_t)c.threads),
                                                           cap / (size_t)R));
        c.ctas = (int)(chunks * (size_t)R);
      } else {
        c.ctas = std::max(R, c.ctas - c.ctas % R);
      }
      break;
    }
    case AR_ONESHOT_FANOUT_BULK: {
      c.threads = ar::kBulkThreads;
      const size_t tiles = ceil_div(groups, (size_t)ar::kBulkThreads);
      const size_t resident = (size_t)h->bulk_ctas_per_sm * (size_t)h->num_sms;
      if (c.ctas <= 0) c.ctas = (int)std::max<size_t>(1, std::min(tiles, resident));
      break;
    }
    case AR_PACKET_3OP: {
      // Three ordinary launches: no co-residency needed, one group per thread.
      if (c.threads <= 0) c.threads = h->fused_threads;
      size_t per_rank = std::max<size_t>(1, ceil_div(shard_groups, (size_t)c.threads));
      if (c.ctas > 0) per_rank = std::max<size_t>(1, (size_t)c.ctas / (size_t)R);
      per_rank = std::min(per_rank, std::max<size_t>(1, cap / (size_t)R));
      c.ctas = (int)(per_rank * (size_t)R);
      break;
    }
    case AR_FUSED_LL8:
    case AR_FUSED_LL8_STAGED: {
      // One clique per CTA: R warp groups of Tr threads; a persistent grid of
      // at most the co-resident CTAs, at most one per tile of Tr groups.
      const int tr = fused_tr(h, variant, c.threads > 0 ? c.threads : h->fused_threads);
      c.threads = R * tr;
      const size_t limit =
          std::max<size_t>(1, (size_t)occupancy(h, variant, c.threads) * (size_t)h->num_sms);
      size_t ctas = c.ctas > 0 ? (size_t)c.ctas : ceil_div(shard_groups, (size_t)tr);
      c.ctas = (int)std::max<size_t>(1, std::min(ctas, limit));
      const FusedMode m = fused_mode(h, shard_groups, tr, variant == AR_FUSED_LL8);
      if (m.ring_rounds) {  // every CTA's ring must fit (at least one does)
        const size_t per_cta = ring_groups_per_cta(R, m.ring_rounds, tr);
        c.ctas = (int)std::max<size_t>(1, std::min((size_t)c.ctas, h->ring_groups / per_cta));
      }
      break;
    }
    default:
      break;
  }
  return c;
}

// Guard zones around every packet region: kGuardBytes of kGuardByte before
// and after it, never touched by the library, checked by
// ar_debug_check_guards (writes outside a region would change them).
constexpr size_t kGuardBytes = 4096;
constexpr unsigned char kGuardByte = 0x5A;

cudaError_t guarded_alloc(size_t bytes, void** region, void** base) {
  char* p = nullptr;
  cudaError_t e = cudaMalloc(&p, bytes + 2 * kGuardBytes);
  if (e != cudaSuccess) return e;
  *base = p;
  if ((e = cudaMemset(p, kGuardByte, kGuardBytes)) != cudaSuccess) return e;
  if ((e = cudaMemset(p + kGuardBytes + bytes, kGuardByte, kGuardBytes)) != cudaSuccess) return e;
  *region = p + kGuardBytes;  // 256-byte aligned like the allocation
  return cudaSuccess;
}

// Writes a temporary buffer of twice the L2 size on the current device and
// waits, so that every dirty line L2 held before (the packet scratch just
// zeroed) has been written back to memory.  The fused kernel drops consumed
// packet lines from L2 without writing them back, after which they read back
// as their memory contents: this makes those contents zeros or packets of
// earlier calls (older flags), never whatever the memory held before.
cudaError_t write_back_l2(int dev) {
  int l2 = 0;
  cudaError_t e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
  if (e != cudaSuccess) return e;
  const size_t bytes = 2 * (size_t)(l2 > 0 ? l2 : (128 << 20));
  void* tmp = nullptr;
  if ((e = cudaMalloc(&tmp, bytes)) != cudaSuccess) return e;
  e = cudaMemset(tmp, 0xA5, bytes);
  const cudaError_t e2 = cudaDeviceSynchronize();
  const cudaError_t e3 = cudaFree(tmp);
  return e != cudaSuccess ? e : e2 != cudaSuccess ? e2 : e3;
}

ar_status_t check_device(const ar_ctx* h) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return AR_ERR_CUDA;
  return dev == h->device ? AR_OK : AR_ERR_INVALID_ARG;
}

ar_status_t launch(ar_ctx* h, int variant, const TuneRow* row, const void* const* d_in,
                   void* const* d_out, size_t count, cudaStream_t s, bool host_memory = false) {
  NvtxRange range(range_name(variant));
  CallArgs a;
  if (is_packet_variant(variant) && h->R > AR_MAX_PACKET_RANKS) return AR_ERR_UNSUPPORTED;
  a.in_tbl = reinterpret_cast<const char* const*>(d_in);
  a.out_tbl = reinterpret_cast<char* const*>(d_out);
  a.count = count;
  a.groups = ceil_div(count, (size_t)ar::group_elems(h->dtype));
  a.shard_groups = ceil_div(a.groups, (size_t)h->R);
  a.state = h->state;
  a.spin_limit_ns = h->spin_limit_ns;
  LaunchCfg cfg = shape(h, variant, row, a.groups, a.shard_groups, host_memory);
  cfg.pdl = h->pdl && 2 * (size_t)h->R * count * h->elem_bytes <=
                         (variant == AR_TWOPHASE ? h->pdl_max_bytes_twophase : h->pdl_max_bytes);
  if (variant == AR_FUSED_LL8 || variant == AR_FUSED_LL8_STAGED) cfg.pdl = h->pdl && h->fused_pdl;
  if (h->log)
    fprintf(stderr, "[ar] R=%d count=%zu variant=%s ctas=%d threads=%d pdl=%d\n", h->R, count,
            ar_variant_name(variant), cfg.ctas, cfg.threads, (int)cfg.pdl);
  if (cfg.ctas <= 0 || cfg.threads <= 0) return AR_ERR_CUDA;
  cudaError_t e = cudaErrorInvalidValue;
  switch (variant) {
    case AR_ONESHOT_PULL:
      e = ar::launch_oneshot_pull(h->R, h->dtype, a, cfg, s);
      break;
    case AR_ONESHOT_FANOUT:
      e = ar::launch_oneshot_fanout(h->R, h->dtype, a, cfg, s);
      break;
    case AR_TWOPHASE:
      e = ar::launch_twophase(h->R, h->dtype, a, cfg, s);
      break;
    case AR_ONESHOT_FANOUT_BULK:
      e = ar::launch_oneshot_fanout_bulk(h->R, h->dtype, a, cfg, s);
      break;
    case AR_FUSED_LL8:
    case AR_FUSED_LL8_STAGED:
    case AR_PACKET_3OP: {
      FusedArgs f;
      f.scratch = h->scratch;
      f.rscratch = h->rscratch;
      f.slot_groups = h->slot_groups;
      f.state = h->state;
      f.spin_limit_ns = h->spin_limit_ns;
      f.skip_producer = h->skip_producer;
      const FusedMode m =
          fused_mode(h, a.shard_groups, cfg.threads / h->R, variant != AR_FUSED_LL8_STAGED);
      f.lead = m.lead;
      f.discard = m.discard;
      f.ring = h->ring;
      f.ring_rounds = variant == AR_FUSED_LL8 ? m.ring_rounds : 0;
      f.fast32 = ar::fused_fits_32bit(h->R, a.shard_groups, h->slot_groups);
      f.delay_rank = h->delay_rank;
      f.delay_ns = h->delay_ns;
      h->skip_producer = -1;
      if (h->log)
        fprintf(stderr, "[ar]   packets: lead=%d discard=%d ring_rounds=%d\n", f.lead, f.discard,
                f.ring_rounds);
      const int dt = h->dtype;
      e = variant == AR_FUSED_LL8          ? ar::launch_fused_ll8(h->R, dt, a, f, cfg, s)
          : variant == AR_FUSED_LL8_STAGED ? ar::launch_fused_ll8_staged(h->R, dt, a, f, cfg, s)
                                           : ar::launch_packet_3op(h->R, dt, a, f, cfg, s);
      break;
    }
    default:
      return AR_ERR_INVALID_ARG;
  }
  return cuda_status(e);
}

}  // namespace

extern "C" {

const char* ar_status_string(int status) {
  switch (status) {
    case AR_OK: return "ok";
    case AR_ERR_INVALID_ARG: return "invalid argument";
    case AR_ERR_UNSUPPORTED: return "unsupported dtype or device";
    case AR_ERR_OOM: return "device out of memory";
    case AR_ERR_CUDA: return "CUDA runtime error";
    case AR_ERR_TIMEOUT: return "packet wait timed out on the device";
    default: return "unknown status";
  }
}

const char* ar_variant_name(int variant) {
  switch (variant) {
    case AR_AUTO: return "auto";
    case AR_ONESHOT_PULL: return "oneshot_pull";
    case AR_ONESHOT_FANOUT: return "oneshot_fanout";
    case AR_TWOPHASE: return "twophase";
    case AR_FUSED_LL8: return "fused_ll8";
    case AR_ONESHOT_FANOUT_BULK: return "oneshot_fanout_bulk";
    case AR_FUSED_LL8_STAGED: return "fused_ll8_staged";
    case AR_PACKET_3OP: return "packet_3op";
    default: return "?";
  }
}

ar_status_t ar_create(int R, size_t max_count, int dtype, ar_handle_t* out) {
  if (!out) return AR_ERR_INVALID_ARG;
  *out = nullptr;
  if (R < 1 || R > AR_MAX_RANKS || max_count == 0) return AR_ERR_INVALID_ARG;
  if (max_count > ((size_t)1 << 40)) return AR_ERR_INVALID_ARG;
  if (dtype != AR_BF16 && dtype != AR_FP16 && dtype != AR_FP32) return AR_ERR_UNSUPPORTED;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return AR_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return AR_ERR_CUDA;
  if (major != 10 || minor != 3) return AR_ERR_UNSUPPORTED;

  ar_ctx* h = new (std::nothrow) ar_ctx();
  if (!h) return AR_ERR_OOM;
  h->R = R;
  h->dtype = dtype;
  h->elem_bytes = dtype == AR_FP32 ? 4 : 2;
  h->max_count = max_count;
  h->device = dev;
  h->num_sms = sms;
  cudaDeviceGetAttribute(&h->l2_bytes, cudaDevAttrL2CacheSize, dev);
  h->table = builtin_table(R, dtype == AR_FP32 ? 4 : 2);
  const char* env = getenv("AR_TUNING_FILE");
  if (env && *env && !load_table_file(env, &h->table)) {
    fprintf(stderr, "[ar] cannot use AR_TUNING_FILE=%s; keeping the built-in table\n", env);
  }
  env = getenv("AR_VARIANT");
  if (env && *env) {
    int v = parse_variant(env);
    if (v >= 0) h->variant = v;
  }
  env = getenv("AR_SPIN_LIMIT_NS");
  if (env && *env) {
    unsigned long long ns = strtoull(env, nullptr, 10);
    if (ns >= 1000) h->spin_limit_ns = ns;
  }
  env = getenv("AR_LOG");
  h->log = env && env[0] == '1';
  env = getenv("AR_PDL");
  if (env && env[0] == '0') h->pdl = false;
  env = getenv("AR_PDL_MAX_MB");
  if (env && *env) {
    const long mb = strtol(env, nullptr, 10);
    if (mb >= 0) h->pdl_max_bytes = (size_t)mb << 20;
  }
  env = getenv("AR_FUSED_LEAD");
  if (env && *env) {
    const long v = strtol(env, nullptr, 10);
    if (v >= 1 && v <= 2) h->fused_lead = (int)v;
  }
  env = getenv("AR_FUSED_RING");
  if (env && (env[0] == '0' || env[0] == '1')) h->fused_ring = env[0] - '0';
  env = getenv("AR_FUSED_PDL");
  if (env && env[0] == '0') h->fused_pdl = false;
  env = getenv("AR_FUSED_DISCARD");
  if (env && (env[0] == '0' || env[0] == '1')) h->fused_discard = env[0] - '0';

  const size_t groups = ceil_div(max_count, (size_t)ar::group_elems(dtype));
  // Rounded up to 4 groups so that every slot starts on a 128-byte line.
  // The packet variants (and their scratch) exist for R <= AR_MAX_PACKET_RANKS.
  const bool packets = R <= AR_MAX_PACKET_RANKS;
  h->slot_groups = (ceil_div(groups, (size_t)R) + 3) / 4 * 4;
  h->scratch_bytes =
      packets ? (size_t)R * (size_t)(R - 1) * h->slot_groups * 4 * sizeof(uint64_t) : 0;
  h->fused_ctas_per_sm =
      packets ? occupancy(h, AR_FUSED_LL8, R * fused_tr(h, AR_FUSED_LL8, h->fused_threads)) : 0;
  if (ar::bulk_prepare(R, dtype) == cudaSuccess) h->bulk_ctas_per_sm = ar::bulk_ctas_per_sm(R, dtype);
  cudaGetLastError();

  ar_status_t st = AR_OK;
  if (cudaMalloc(&h->state, sizeof(DevState)) != cudaSuccess) st = AR_ERR_OOM;
  if (st == AR_OK && h->scratch_bytes) {
    void* r0 = nullptr;
    void* r1 = nullptr;
    if (guarded_alloc(h->scratch_bytes, &r0, &h->region_base[0]) != cudaSuccess ||
        guarded_alloc(h->scratch_bytes, &r1, &h->region_base[1]) != cudaSuccess)
      st = AR_ERR_OOM;
    h->scratch = static_cast<uint64_t*>(r0);
    h->rscratch = static_cast<uint64_t*>(r1);
    h->region_bytes[0] = h->region_bytes[1] = h->scratch_bytes;
  }
  if (st == AR_OK) {
    DevState init;
    memset(&init, 0, sizeof init);
    init.epoch = 1;
    if (cudaMemcpy(h->state, &init, sizeof init, cudaMemcpyHostToDevice) != cudaSuccess)
      st = AR_ERR_CUDA;
  }
  if (st == AR_OK && h->scratch_bytes &&
      (cudaMemset(h->scratch, 0, h->scratch_bytes) != cudaSuccess ||
       cudaMemset(h->rscratch, 0, h->scratch_bytes) != cudaSuccess))
    st = AR_ERR_CUDA;
  // The fused kernel's rings: room for every co-resident CTA at the default
  // and at the largest CTA size, no more than the message needs.
  if (st == AR_OK && packets && R > 1) {
    size_t cap = 0;
    for (int threads : {h->fused_threads, 512}) {
      const int tr = fused_tr(h, AR_FUSED_LL8, threads);
      const size_t ctas = std::min((size_t)occupancy(h, AR_FUSED_LL8, R * tr) * (size_t)sms,
                                   ceil_div(h->slot_groups, (size_t)tr));
      cap = std::max(cap, ctas * ring_groups_per_cta(R, kMaxRingRounds, tr));
    }
    h->ring_groups = cap;
    void* r2 = nullptr;
    if (cap && (guarded_alloc(cap * 32, &r2, &h->region_base[2]) != cudaSuccess ||
                cudaMemset(r2, 0, cap * 32) != cudaSuccess))
      st = AR_ERR_OOM;
    h->ring = static_cast<uint64_t*>(r2);
    h->region_bytes[2] = cap * 32;
  }
  if (st == AR_OK && cudaDeviceSynchronize() != cudaSuccess) st = AR_ERR_CUDA;
  if (st == AR_OK && h->scratch_bytes && h->fused_discard != 0 && write_back_l2(dev) != cudaSuccess)
    st = AR_ERR_OOM;
  if (st != AR_OK) {
    cudaGetLastError();
    ar_destroy(h);
    return st;
  }
  *out = h;
  return AR_OK;
}

ar_status_t ar_destroy(ar_handle_t h) {
  if (!h) return AR_OK;
  ar_status_t st = AR_OK;
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != h->device) cudaSetDevice(h->device);
  if (cudaDeviceSynchronize() != cudaSuccess) st = AR_ERR_CUDA;
  for (void* b : h->region_base)
    if (b && cudaFree(b) != cudaSuccess) st = AR_ERR_CUDA;
  if (h->state && cudaFree(h->state) != cudaSuccess) st = AR_ERR_CUDA;
  if (h->staging && cudaFree(h->staging) != cudaSuccess) st = AR_ERR_CUDA;
  if (h->staging_tables && cudaFree(h->staging_tables) != cudaSuccess) st = AR_ERR_CUDA;
  if (h->direct_tables && cudaFree(h->direct_tables) != cudaSuccess) st = AR_ERR_CUDA;
  if (prev >= 0 && prev != h->device) cudaSetDevice(prev);
  delete h;
  return st;
}

ar_status_t ar_set_variant(ar_handle_t h, int variant) {
  if (!h || variant < 0 || variant >= AR_NUM_VARIANTS) return AR_ERR_INVALID_ARG;
  h->variant = variant;
  return AR_OK;
}

ar_status_t ar_select(ar_handle_t h, size_t count, int* variant) {
  if (!h || !variant) return AR_ERR_INVALID_ARG;
  const TuneRow* row = nullptr;
  *variant = choose(h, count, &row);
  return AR_OK;
}

ar_status_t ar_set_launch(ar_handle_t h, int variant, int ctas, int threads) {
  if (!h || variant <= AR_AUTO || variant >= AR_NUM_VARIANTS) return AR_ERR_INVALID_ARG;
  if (ctas < 0 || threads < 0) return AR_ERR_INVALID_ARG;
  if (threads && (threads % 32 || threads < 64 || threads > 512)) return AR_ERR_INVALID_ARG;
  if ((variant == AR_FUSED_LL8 || variant == AR_ONESHOT_FANOUT) && threads &&
      (threads < 128 || threads > 512))
    return AR_ERR_INVALID_ARG;
  h->override_cfg[variant] = {ctas, threads};
  return AR_OK;
}

ar_status_t ar_set_spin_limit_ns(ar_handle_t h, uint64_t ns) {
  if (!h || ns < 1000) return AR_ERR_INVALID_ARG;
  h->spin_limit_ns = ns;
  return AR_OK;
}

ar_status_t ar_query(ar_handle_t h, ar_info_t* info) {
  if (!h || !info) return AR_ERR_INVALID_ARG;
  info->R = h->R;
  info->dtype = h->dtype;
  info->max_count = h->max_count;
  info->scratch_bytes = 2 * h->scratch_bytes + h->ring_groups * 32;
  info->num_sms = h->num_sms;
  info->fused_max_ctas = h->fused_ctas_per_sm * h->num_sms;
  info->fused_threads = h->R * fused_tr(h, AR_FUSED_LL8, h->fused_threads);
  info->device = h->device;
  return AR_OK;
}

ar_status_t ar_allreduce(ar_handle_t h, const void* const* d_in_tbl, void* const* d_out_tbl,
                         size_t count, void* stream) {
  if (!h || !d_in_tbl || !d_out_tbl) return AR_ERR_INVALID_ARG;
  if (count > h->max_count) return AR_ERR_INVALID_ARG;
  if (count == 0) return AR_OK;
  ar_status_t st = check_device(h);
  if (st != AR_OK) return st;
  const TuneRow* row = nullptr;
  const int v = choose(h, count, &row);
  return launch(h, v, row, d_in_tbl, d_out_tbl, count, static_cast<cudaStream_t>(stream));
}

// Reduce-scatter (rs = true) or all-gather of blocks of `block` elements.
static ar_status_t launch_block_collective(ar_handle_t h, bool rs, const void* const* d_in,
                                           void* const* d_out, size_t block, void* stream) {
  if (!h || !d_in || !d_out) return AR_ERR_INVALID_ARG;
  if (block == 0) return AR_OK;
  if (block > h->max_count / (size_t)h->R) return AR_ERR_INVALID_ARG;
  NvtxRange range(rs ? "ar reduce_scatter" : "ar all_gather");
  ar_status_t st = check_device(h);
  if (st != AR_OK) return st;
  CallArgs a;
  a.in_tbl = reinterpret_cast<const char* const*>(d_in);
  a.out_tbl = reinterpret_cast<char* const*>(d_out);
  a.count = block;
  a.groups = ceil_div(block, (size_t)ar::group_elems(h->dtype));
  a.shard_groups = a.groups;
  a.state = h->state;
  a.spin_limit_ns = h->spin_limit_ns;
  LaunchCfg cfg;
  cfg.threads = 256;
  const size_t cap = std::max<size_t>(1, (size_t)h->num_sms * 16 / (size_t)h->R);
  cfg.ctas = (int)std::max<size_t>(1, std::min(ceil_div(a.groups, (size_t)cfg.threads), cap));
  cfg.pdl = h->pdl && (size_t)h->R * (h->R + 1) * block * h->elem_bytes <= h->pdl_max_bytes;
  if (h->log)
    fprintf(stderr, "[ar] R=%d %s block=%zu ctas=%dx%d threads=%d\n", h->R,
            rs ? "reduce_scatter" : "all_gather", block, cfg.ctas, h->R, cfg.threads);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(rs ? ar::launch_reduce_scatter(h->R, h->dtype, a, cfg, s)
                        : ar::launch_all_gather(h->R, h->dtype, a, cfg, s));
}

ar_status_t ar_reduce_scatter(ar_handle_t h, const void* const* d_in_tbl, void* const* d_out_tbl,
                              size_t recvcount, void* stream) {
  return launch_block_collective(h, true, d_in_tbl, d_out_tbl, recvcount, stream);
}

ar_status_t ar_all_gather(ar_handle_t h, const void* const* d_in_tbl, void* const* d_out_tbl,
                          size_t sendcount, void* stream) {
  return launch_block_collective(h, false, d_in_tbl, d_out_tbl, sendcount, stream);
}

ar_status_t ar_get_device_status(ar_handle_t h, void* stream) {
  if (!h) return AR_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Bounded poll instead of an unbounded synchronise.
  const int max_polls = 600000;  // 60 s at 100 us
  int polls = 0;
  cudaError_t q;
  while ((q = cudaStreamQuery(s)) == cudaErrorNotReady) {
    if (++polls > max_polls) return AR_ERR_CUDA;
    struct timespec ts = {0, 100000};
    nanosleep(&ts, nullptr);
  }
  if (q != cudaSuccess) return AR_ERR_CUDA;
  DevState host;
  if (cudaMemcpy(&host, h->state, sizeof host, cudaMemcpyDeviceToHost) != cudaSuccess)
    return AR_ERR_CUDA;
  if (host.error == ar::kDevErrNone) return AR_OK;
  h->last_error = host.error;
  h->last_error_info = host.error_info;
  h->last_timeouts = host.timeouts;
  const uint32_t zero[3] = {0, 0, 0};  // error, error_info, timeouts
  if (cudaMemcpy(&h->state->error, zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return AR_ERR_CUDA;
  return host.error == ar::kDevErrTimeout ? AR_ERR_TIMEOUT : AR_ERR_CUDA;
}

ar_status_t ar_debug_check_guards(ar_handle_t h, int* intact) {
  if (!h || !intact) return AR_ERR_INVALID_ARG;
  *intact = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return AR_ERR_CUDA;
  std::vector<unsigned char> buf(kGuardBytes);
  for (int i = 0; i < 3; ++i) {
    if (!h->region_base[i]) continue;
    const char* base = static_cast<const char*>(h->region_base[i]);
    for (const char* g : {base, base + kGuardBytes + h->region_bytes[i]}) {
      if (cudaMemcpy(buf.data(), g, kGuardBytes, cudaMemcpyDeviceToHost) != cudaSuccess)
        return AR_ERR_CUDA;
      for (unsigned char c : buf)
        if (c != kGuardByte) return AR_OK;
    }
  }
  *intact = 1;
  return AR_OK;
}

ar_status_t ar_last_timeout(ar_handle_t h, int* waiting_rank, int* missing_rank,
                            uint32_t* waits) {
  if (!h || !waiting_rank || !missing_rank || !waits) return AR_ERR_INVALID_ARG;
  if (h->last_error != ar::kDevErrTimeout) {
    *waiting_rank = -1;
    *missing_rank = -1;
    *waits = 0;
    return AR_OK;
  }
  *waiting_rank = (int)(h->last_error_info >> 16);
  const uint32_t m = h->last_error_info & 0xFFFFu;
  *missing_rank = m == 0xFFFFu ? -1 : (int)m;
  *waits = h->last_timeouts;
  return AR_OK;
}

ar_status_t ar_reserve_host_staging(ar_handle_t h) {
  if (!h) return AR_ERR_INVALID_ARG;
  if (h->staging) return AR_OK;
  const size_t per_rank = (h->max_count + 127) / 128 * 128;  // keep every buffer 256-byte aligned
  const size_t elems = 2 * (size_t)h->R * per_rank;
  if (cudaMalloc(&h->staging, elems * h->elem_bytes) != cudaSuccess) {
    cudaGetLastError();
    h->staging = nullptr;
    return AR_ERR_OOM;
  }
  if (cudaMalloc(&h->staging_tables, 2 * (size_t)h->R * sizeof(char*)) != cudaSuccess ||
      cudaMalloc(&h->direct_tables, 2 * (size_t)h->R * sizeof(char*)) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->staging);
    if (h->staging_tables) cudaFree(h->staging_tables);
    h->staging = nullptr;
    h->staging_tables = nullptr;
    h->direct_tables = nullptr;
    return AR_ERR_OOM;
  }
  std::vector<char*> ptrs(2 * (size_t)h->R);
  for (size_t i = 0; i < ptrs.size(); ++i) ptrs[i] = h->staging + i * per_rank * h->elem_bytes;
  if (cudaMemcpy(h->staging_tables, ptrs.data(), ptrs.size() * sizeof(char*),
                 cudaMemcpyHostToDevice) != cudaSuccess)
    return AR_ERR_CUDA;
  return AR_OK;
}

ar_status_t ar_allreduce_host(ar_handle_t h, const void* const* h_in, void* const* h_out,
                              size_t count, void* stream) {
  if (!h || !h_in || !h_out || !h->staging) return AR_ERR_INVALID_ARG;
  if (count > h->max_count) return AR_ERR_INVALID_ARG;
  if (count == 0) return AR_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Not capturable: the direct path's pointer table is copied from this
  // call's stack (a captured copy node would keep pointing at it), and the
  // staging path copies from pageable memory.  Refuse before any other work.
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &capture) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  if (capture != cudaStreamCaptureStatusNone) return AR_ERR_UNSUPPORTED;
  ar_status_t st = check_device(h);
  if (st != AR_OK) return st;
  NvtxRange range("ar allreduce_host");
  for (int r = 0; r < h->R; ++r)
    if (!h_in[r] || !h_out[r]) return AR_ERR_INVALID_ARG;

  // Direct path: page-locked host buffers (and device buffers) are
  // addressable by the kernels through unified addressing -- over
  // NVLink-C2C on Grace-Blackwell -- so the kernel itself reads every input
  // byte from the host once and writes every output byte to the host once,
  // both directions at the same time.  The pointer table goes to the device
  // in stream order (copied out of this stack array before the call returns).
  void* direct[2 * AR_MAX_RANKS];
  // The bulk-copy variant keeps to device memory (staging path).
  bool ok_direct = h->variant != AR_ONESHOT_FANOUT_BULK;
  for (int i = 0; i < 2 * h->R && ok_direct; ++i) {
    const void* p = i < h->R ? h_in[i] : h_out[i - h->R];
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      cudaGetLastError();
      ok_direct = false;
    } else if ((at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeDevice ||
                at.type == cudaMemoryTypeManaged) &&
               at.devicePointer != nullptr) {
      direct[i] = at.devicePointer;
    } else {
      ok_direct = false;
    }
  }
  if (ok_direct) {
    if (cudaMemcpyAsync(h->direct_tables, direct, 2 * (size_t)h->R * sizeof(void*),
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
      return AR_ERR_CUDA;
    // The fan-out reads and writes each byte exactly once: the selector's
    // choice for host memory unless a variant is forced.
    const int v = h->variant != AR_AUTO ? h->variant : AR_ONESHOT_FANOUT;
    return launch(h, v, nullptr, reinterpret_cast<const void* const*>(h->direct_tables),
                  reinterpret_cast<void* const*>(h->direct_tables + h->R), count, s,
                  /*host_memory=*/true);
  }

  // Staging path (pageable host memory): one copy per rank each way.
  const size_t per_rank = (h->max_count + 127) / 128 * 128;
  const size_t bytes = count * h->elem_bytes;
  for (int r = 0; r < h->R; ++r) {
    if (cudaMemcpyAsync(h->staging + (size_t)r * per_rank * h->elem_bytes, h_in[r], bytes,
                        cudaMemcpyHostToDevice,
                        s) != cudaSuccess)
      return AR_ERR_CUDA;
  }
  const TuneRow* row = nullptr;
  const int v = choose(h, count, &row);
  st = launch(h, v, row, reinterpret_cast<const void* const*>(h->staging_tables),
              reinterpret_cast<void* const*>(h->staging_tables + h->R), count, s);
  if (st != AR_OK) return st;
  for (int r = 0; r < h->R; ++r) {
    if (cudaMemcpyAsync(h_out[r], h->staging + (size_t)(h->R + r) * per_rank * h->elem_bytes, bytes,
                        cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return AR_ERR_CUDA;
  }
  return AR_OK;
}

ar_status_t ar_debug_skip_producer(ar_handle_t h, int rank) {
  if (!h || rank < -1 || rank >= h->R) return AR_ERR_INVALID_ARG;
  h->skip_producer = rank;
  return AR_OK;
}

ar_status_t ar_debug_delay_producer(ar_handle_t h, int rank, uint64_t ns) {
  if (!h || rank < -1 || rank >= h->R || ns > 10ull * 1000ull * 1000ull) return AR_ERR_INVALID_ARG;
  h->delay_rank = ns ? rank : -1;
  h->delay_ns = rank >= 0 ? ns : 0;
  return AR_OK;
}

ar_status_t ar_debug_set_epoch(ar_handle_t h, uint32_t epoch) {
  if (!h || epoch == 0) return AR_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return AR_ERR_CUDA;
  // A jump of the epoch invalidates the "older flag = not arrived" ordering
  // for everything written before it: clear every packet.
  if ((h->scratch_bytes && (cudaMemset(h->scratch, 0, h->scratch_bytes) != cudaSuccess ||
                            cudaMemset(h->rscratch, 0, h->scratch_bytes) != cudaSuccess)) ||
      (h->ring && cudaMemset(h->ring, 0, h->ring_groups * 32) != cudaSuccess) ||
      cudaDeviceSynchronize() != cudaSuccess)
    return AR_ERR_CUDA;
  if (h->scratch_bytes && h->fused_discard != 0 && write_back_l2(h->device) != cudaSuccess)
    return AR_ERR_CUDA;
  return cuda_status(cudaMemcpy(&h->state->epoch, &epoch, sizeof epoch, cudaMemcpyHostToDevice));
}

ar_status_t ar_debug_get_epoch(ar_handle_t h, uint32_t* epoch) {
  if (!h || !epoch) return AR_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return AR_ERR_CUDA;
  return cuda_status(cudaMemcpy(epoch, &h->state->epoch, sizeof *epoch, cudaMemcpyDeviceToHost));
}

}  // extern "C"
