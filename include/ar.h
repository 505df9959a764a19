/*
 * ar.h -- C ABI of the GB300 virtual-rank allreduce library
 *         (libar_gb300.so).
 *
 * R "virtual ranks" are R separate buffers in the HBM of ONE GPU.  An
 * allreduce leaves, in every rank's output buffer, the element-wise sum of
 * all R input buffers:
 *
 *     out_r[i] = rne( ((float)in_0[i] + (float)in_1[i]) + ... + (float)in_{R-1}[i] )
 *
 * for every r in [0, R) and i in [0, count): fp32 additions in rank order
 * 0..R-1 (seeded with rank 0's value, no fused multiply-add), one final
 * round-to-nearest-even to the element type (bf16 or fp16; none for fp32).
 * Every variant below produces this result bit for bit; they differ only in
 * how the data moves.
 *
 * Where each operation comes from:
 *   - the input/output pointer tables mirror the broadcast table of output
 *     pointers of "optimize allreduce write mode by broadcast output ptr"
 *     (ROCm/aiter #1910, Motivation and Technical Details) and the device
 *     array of peer pointers passed as a kernel argument in "One shot all
 *     reduce Example" (pytorch-labs/helion #245, review discussion);
 *   - AR_ONESHOT_PULL is the one-shot allreduce of "One shot all reduce
 *     Example" (every rank reads all peers and reduces locally);
 *   - AR_ONESHOT_FANOUT is that one-shot read combined with the write mode of
 *     the aiter page (the reduced value is written straight into every
 *     rank's output through the output-pointer table);
 *   - AR_TWOPHASE is the two-stage allreduce of the aiter page without write
 *     mode (stage 1 reduces a shard into its owner's output, stage 2 copies
 *     it into the other ranks' outputs);
 *   - AR_ONESHOT_FANOUT_BULK is the same fan-out with every input tile
 *     brought into shared memory, and every result tile sent to the R
 *     outputs, by the bulk-copy (TMA) engine;
 *   - AR_FUSED_LL8_STAGED is the fused kernel below without write mode,
 *     otherwise the same kernel: each owner sends its reduced shard back as
 *     LL8 packets to every rank's result slot and every rank copies them
 *     into its output (the packet broadcast of the ARK page);
 *     AR_PACKET_3OP runs the three phases as three launches over the whole
 *     message (that page's send_packet -> recv_reduce_send_packet ->
 *     recv_packet decomposition).  Both exist to measure what write mode
 *     and fusion save;
 *   - AR_FUSED_LL8 is the single fused scatter -> reduce -> broadcast kernel
 *     synchronised by LL packet flags of "Add monolithic fused packet
 *     allreduce kernel and Model::all_reduce_packet API" (microsoft/ark #254,
 *     Changes), with the flag rotated on every call (that page's Known
 *     limitations leave Flag = 1 hardcoded), and the broadcast done in the
 *     aiter write mode.  Each CTA holds one warp group per virtual rank, so
 *     packet exchanges stay within a CTA and no CTA waits on another (the
 *     page's NumProcs >= NPeers limitation cannot arise); the kernel is
 *     pipelined over rounds so that its packets stay in L2.
 *
 * Threading: a handle may be used from one host thread at a time.  Calls on
 * one handle must be ordered on one stream (one call in flight), because a
 * handle owns one packet scratch region and one epoch; use one handle per
 * concurrent stream.  (The one-shot region of "Add HIP-graph capture
 * coverage for the sharded-relay collectives" (meta-pytorch/torchcomms
 * #3850, region-lifetime commit) has the same precondition.)
 *
 * Launch overlap: the one-shot, two-phase, bulk fan-out, reduce-scatter and
 * all-gather kernels of a call that moves at most 16 MiB (two-phase: 8 MiB)
 * are launched with programmatic dependent launch, so they may be scheduled
 * while the previous kernel in the stream is still running; each waits for that kernel to
 * complete (and its writes to be visible) before touching global memory, so
 * results are those of plain stream order.  The environment variable
 * AR_PDL=0, read by ar_create, turns this off.  The two pipelined fused
 * kernels (AR_FUSED_LL8, AR_FUSED_LL8_STAGED) are launched this way at every
 * size unless AR_PDL=0 or AR_FUSED_PDL=0; the three-launch packet form never
 * is.  Such a kernel reads the two pointer tables (not the buffers they
 * point to) before that wait, so the table round trip overlaps the previous
 * kernel's tail.  Hence a precondition: the tables must not be written by
 * the kernel just before the call in the same stream if that kernel lets
 * its dependents start early (griddepcontrol.launch_dependents) before it
 * writes them.  Tables written by a copy, a memset, any kernel without such
 * a trigger, or an earlier call of this library (which never writes them)
 * are safe.
 *
 * Streams are passed as `void*` holding a cudaStream_t (NULL = the legacy
 * default stream), so that this header needs no CUDA header.
 */
#ifndef AR_GB300_H
#define AR_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define AR_MAX_RANKS 16        /* one-shot, two-phase, reduce-scatter, all-gather */
#define AR_MAX_PACKET_RANKS 8  /* the LL8 packet variants */

typedef struct ar_ctx* ar_handle_t;

typedef enum {
  AR_BF16 = 0, /* bfloat16, 2 bytes: fp32 accumulation, one round to nearest even */
  AR_FP16 = 1, /* IEEE binary16, 2 bytes: fp32 accumulation, one round to nearest even */
  AR_FP32 = 2  /* IEEE binary32, 4 bytes: fp32 accumulation, no final rounding */
} ar_dtype_t;

typedef enum {
  AR_OK = 0,
  AR_ERR_INVALID_ARG = 1, /* bad R, count, pointer, variant or handle */
  AR_ERR_UNSUPPORTED = 2, /* unknown dtype, a packet variant with R > 8, no sm_103 device,
                             or ar_allreduce_host under stream capture */
  AR_ERR_OOM = 3,         /* device allocation failed in ar_create */
  AR_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, copy, sync) */
  AR_ERR_TIMEOUT = 5      /* a packet wait inside the fused kernel gave up */
} ar_status_t;

typedef enum {
  AR_AUTO = 0,           /* per-size selector (measured table) picks one of the below */
  AR_ONESHOT_PULL = 1,   /* CTA (chunk, r) reads all R inputs, writes out_r only */
  AR_ONESHOT_FANOUT = 2, /* CTA reads all R inputs once, writes all R outputs */
  AR_TWOPHASE = 3,       /* launch 1: owner shards reduced; launch 2: shards copied out */
  AR_FUSED_LL8 = 4,      /* one persistent kernel: LL8 packet scatter, poll+reduce, write mode */
  AR_ONESHOT_FANOUT_BULK = 5, /* fan-out with tiles moved by bulk (TMA) copies through shared memory */
  AR_FUSED_LL8_STAGED = 6,    /* fused LL8 without write mode: result packets back to every rank */
  AR_PACKET_3OP = 7           /* the same three packet phases as three separate launches */
} ar_variant_t;

#define AR_NUM_VARIANTS 8

/* Static description of a handle (filled by ar_query). */
typedef struct {
  int R;                    /* virtual ranks */
  int dtype;                /* ar_dtype_t */
  size_t max_count;         /* largest count accepted by ar_allreduce */
  size_t scratch_bytes;     /* LL8 packet scratch owned by the handle (both regions) */
  int num_sms;              /* SMs of the device the handle lives on */
  int fused_max_ctas;       /* co-resident CTA limit used to size the fused grid */
  int fused_threads;        /* threads per CTA of the fused kernel (R warp groups) */
  int device;               /* CUDA device ordinal */
} ar_info_t;

/*
 * ar_create -- make a handle for R virtual ranks of up to `max_count`
 * elements each, on the current CUDA device.
 *   R          1 .. AR_MAX_RANKS (the LL8 packet variants need R <=
 *              AR_MAX_PACKET_RANKS; their scratch is allocated only then).
 *   max_count  >= 1; bounds `count` of later calls and sizes the scratch.
 *   dtype      AR_BF16, AR_FP16 or AR_FP32 (element type of every buffer).
 *   out        receives the handle (set to NULL on failure).
 * Allocates, on the current device, two packet scratch regions (scatter
 * packets and the staged variants' result packets), each
 * 32 * R * (R-1) * S bytes with S = ceil(ceil(max_count/G)/R) rounded up
 * to a multiple of 4, G = 8 elements per 16-byte group for bf16/fp16 and 4
 * for fp32 (about 4*(R-1)*max_count bytes for 2-byte types), zeroed here
 * so that no flag matches a live epoch, then written back from L2 to memory
 * (the fused kernel drops consumed packet lines from L2 without writing
 * them back, so they read back as these zeros or as older packets; the
 * write-back writes a temporary buffer of twice the L2 size, about 256 MB,
 * freed before ar_create returns, unless AR_FUSED_DISCARD=0); the fused
 * kernel's per-CTA packet rings (3 rounds of (R-1)*32 bytes per co-resident
 * thread, about 52 MB at R = 8, less for small max_count); and
 * a small state block (epoch, done counter, error word).  Synchronous; not
 * for stream capture.
 * Errors: AR_ERR_INVALID_ARG (R, max_count, out), AR_ERR_UNSUPPORTED (dtype,
 * or the current device is not compute capability 10.3), AR_ERR_OOM, AR_ERR_CUDA.
 * Source: the one-shot region of "Add HIP-graph capture coverage for the
 * sharded-relay collectives" (meta-pytorch/torchcomms #3850, the commit that
 * ties the region's lifetime to its communicator: created once with it, never
 * re-created while it lives, so the epoch never resets); scratch and peer
 * references set up once by Model::all_reduce_packet in "Add monolithic fused
 * packet allreduce kernel and Model::all_reduce_packet API" (microsoft/ark
 * #254, Changes).
 */
ar_status_t ar_create(int R, size_t max_count, int dtype, ar_handle_t* out);

/*
 * ar_allreduce -- out_r[i] = rne(sum over s in rank order of in_s[i])
 * for every r < R and i < count.
 *   h          handle from ar_create.
 *   d_in_tbl   DEVICE pointer to an array of R device pointers (8 bytes each,
 *              e.g. a CUDA int64 tensor of data_ptr()s); entry r is rank r's
 *              input buffer of `count` elements of the handle's dtype.
 *   d_out_tbl  DEVICE pointer to an array of R device pointers; entry r is
 *              rank r's output buffer of `count` elements.
 *   count      elements per rank, 0 .. max_count.  0 returns AR_OK, no launch.
 *   stream     cudaStream_t (as void*) the kernels are launched on.
 * The caller owns the buffers and both tables; they must stay valid and
 * unmodified until the call has completed on `stream`.  The kernels read the
 * tables on the device, so the host never dereferences them.
 * Aliasing: out_r may be exactly in_r (in place) for every variant, and any
 * output may alias any input exactly in AR_ONESHOT_FANOUT.  AR_ONESHOT_PULL
 * detects exact aliasing on the device and then writes every output from
 * one CTA per chunk.  Partially overlapping buffers are undefined.
 * Alignment: buffers 16-byte aligned take 16-byte vector loads and stores
 * (AR_ONESHOT_FANOUT: 32-byte ones for calls of at least 4 MiB per rank
 * when every pointer is 32-byte aligned and R <= 8); any misaligned pointer
 * switches that call to element-sized accesses (same result, slower),
 * decided on the device.
 * Allocates nothing, synchronises nothing, so it can be captured into a CUDA
 * graph; the fused kernel's epoch lives on the device and rotates on every
 * execution, including graph replays (by one per call, or, when the kernel
 * keeps its packets in per-CTA rings -- more than two L2 sizes of packets -- by
 * its number of rounds, one flag per round).
 * Errors: AR_ERR_INVALID_ARG (NULL handle or table, count > max_count),
 * AR_ERR_UNSUPPORTED (a packet variant forced with R > 8), AR_ERR_CUDA
 * (launch failure).  A packet wait that exceeds the spin limit
 * is reported later by ar_get_device_status (the outputs of that call are
 * then undefined).
 * Source: the allreduce with every rank's output pointer available inside
 * the kernel, broadcast once on the host in graph mode, of "optimize
 * allreduce write mode by broadcast output ptr" (ROCm/aiter #1910,
 * Motivation and Technical Details); the device array of peer pointers passed
 * as a kernel argument in "One shot all reduce Example" (pytorch-labs/helion
 * #245, review discussion); the fused kernel of microsoft/ark #254, Changes.
 */
ar_status_t ar_allreduce(ar_handle_t h, const void* const* d_in_tbl,
                         void* const* d_out_tbl, size_t count, void* stream);

/*
 * ar_reduce_scatter -- rank r keeps block r of the sum:
 *   out_r[j] = rne(sum over s in rank order of in_s[r*recvcount + j]),
 * j < recvcount.  Same numerics as ar_allreduce.  Each input holds
 * R*recvcount elements, each output recvcount elements; R*recvcount <=
 * max_count.  It is the one-shot push-reduce kernel of "Add HIP-graph
 * capture coverage for the sharded-relay collectives" (meta-pytorch/
 * torchcomms #3850) with a per-peer source stride of one block and an owner
 * offset of the rank's slot times one block; its allreduce case is the one
 * with a stride of zero.
 * ar_all_gather -- every output is the concatenation of all inputs in rank
 * order: out_r[s*sendcount + j] = in_s[j]; inputs hold sendcount elements,
 * outputs R*sendcount; R*sendcount <= max_count.
 * Both: device pointer tables as in ar_allreduce; outputs must not overlap
 * inputs; 16-byte vectors when every pointer is 16-byte aligned and the
 * block length is a multiple of the 16-byte group (8 elements of 2 bytes,
 * 4 of fp32), else element-sized accesses; one launch, no
 * allocation, no synchronisation.  Errors: AR_ERR_INVALID_ARG (NULL handle
 * or table, block too large), AR_ERR_CUDA (launch).  A block of 0 returns
 * AR_OK without a launch.
 */
ar_status_t ar_reduce_scatter(ar_handle_t h, const void* const* d_in_tbl,
                              void* const* d_out_tbl, size_t recvcount, void* stream);
ar_status_t ar_all_gather(ar_handle_t h, const void* const* d_in_tbl,
                          void* const* d_out_tbl, size_t sendcount, void* stream);

/* ar_destroy -- synchronise the device and free everything the handle owns.
 * NULL is accepted.  Returns AR_ERR_CUDA if a free failed.
 * Source: the region freed together with its communicator in the
 * region-lifetime commit of meta-pytorch/torchcomms #3850 (never freeing
 * leaked a region per communicator). */
ar_status_t ar_destroy(ar_handle_t h);

/* ar_set_variant -- force a variant for later calls on h (AR_AUTO restores
 * the selector).  AR_ERR_INVALID_ARG for an unknown value.
 * Source: the per-size choice between schedules at measured crossovers of
 * meta-pytorch/torchcomms #3850 (the commit re-measuring the relay/direct
 * crossovers), and the fixed block size that cost helion #245's one-shot
 * kernel at 1m (performance table note). */
ar_status_t ar_set_variant(ar_handle_t h, int variant);

/* ar_select -- the variant a call of `count` elements would run (the forced
 * one, or the selector's choice under AR_AUTO).  Host-only, no device work. */
ar_status_t ar_select(ar_handle_t h, size_t count, int* variant);

/* ar_set_launch -- override the CTA count and threads per CTA of a variant
 * (0 = automatic).  For AR_FUSED_LL8 and AR_FUSED_LL8_STAGED ctas is the
 * number of CTAs (each one clique of R warp groups), clamped to the
 * co-resident limit (and, in ring mode, to the packet rings' room), and
 * threads is rounded to R warp groups of a multiple of 32 threads each (at
 * least 32), narrowed where the kernel is compiled for fewer (AR_FUSED_LL8
 * for R <= 4 launches at most 256 threads); for the other variants ctas is
 * the grid (the grid-stride CTA
 * count; a multiple of R for the pull, two-phase and three-launch packet
 * kernels).  threads must be a multiple of 32 in [64, 512]
 * (the packet and fan-out kernels accept 128..512). */
ar_status_t ar_set_launch(ar_handle_t h, int variant, int ctas, int threads);

/* ar_set_spin_limit_ns -- the longest a fused-kernel packet wait may spin
 * before it gives up and sets the device error word (default 100 ms,
 * minimum 1000 ns).  Read by each later launch. */
ar_status_t ar_set_spin_limit_ns(ar_handle_t h, uint64_t ns);

/* ar_get_device_status -- wait (bounded: at most 60 s of polling) for
 * `stream` to drain, then read and clear the handle's device error word.
 * AR_OK, AR_ERR_TIMEOUT if some fused call since the last check gave up
 * waiting for packets, AR_ERR_CUDA if the stream did not drain or a copy
 * failed.
 * Source: the stream synchronise replaced by a bounded poll, so that a kernel
 * that never retires is reported instead of hanging, in the summary of
 * meta-pytorch/torchcomms #3850. */
ar_status_t ar_get_device_status(ar_handle_t h, void* stream);

/* ar_last_timeout -- details of the last AR_ERR_TIMEOUT that
 * ar_get_device_status returned on this handle (host-only, no device work):
 * *waiting_rank = the virtual rank whose packet wait gave up first,
 * *missing_rank = the lowest-numbered rank whose packets (scatter packets,
 * or result packets without write mode) it was still missing, *waits = how
 * many waits gave up before the others saw the call abandoned.  Waits for
 * result packets run twice the spin limit, so when a producer stores nothing
 * it is a wait for that producer's scatter packets that runs out first and
 * the producer that is named.  All -1 / 0
 * if no timeout has been reported.  AR_ERR_INVALID_ARG for a NULL argument.
 * Source: no counterpart on the pages; it names the peer that a bounded poll
 * (the summary of meta-pytorch/torchcomms #3850) gave up on, which a
 * multi-GPU caller would use to tell a dead peer from a slow one. */
ar_status_t ar_last_timeout(ar_handle_t h, int* waiting_rank, int* missing_rank,
                            uint32_t* waits);

/* ar_query -- fill *info. */
ar_status_t ar_query(ar_handle_t h, ar_info_t* info);

/* ar_status_string -- static, never NULL.
 * Source: the pages define no such function; it names the status codes
 * above, whose failure modes (a wait that never ends, reported rather than
 * hung on) come from the summary of meta-pytorch/torchcomms #3850. */
const char* ar_status_string(int status);

/* ar_variant_name -- static name of a variant ("auto", "oneshot_pull", ...),
 * "?" for an unknown value. */
const char* ar_variant_name(int variant);

/* ---- host-buffer path (end-to-end use from host memory) ----------------
 *
 * ar_reserve_host_staging -- allocate, once, R input and R output device
 * buffers of max_count elements plus their device pointer tables, used by
 * ar_allreduce_host.  Synchronous.  AR_ERR_OOM / AR_ERR_CUDA on failure.
 *
 * ar_allreduce_host -- h_in[r] / h_out[r] are HOST pointers (host arrays of
 * R host pointers).  When every buffer is page-locked (or device memory),
 * the kernel reads and writes the buffers where they are -- page-locked
 * host memory is device-addressable through unified addressing, over
 * NVLink-C2C on Grace-Blackwell -- so each input byte crosses to the device
 * once and each output byte back once, both directions concurrently; with
 * AR_AUTO this path runs AR_ONESHOT_FANOUT (one read and one write per
 * byte), otherwise the forced variant (AR_ONESHOT_FANOUT_BULK always
 * takes the staging path).  Otherwise (pageable memory) on
 * `stream`: one cudaMemcpyAsync per rank into the staging inputs, the
 * allreduce (same selection as ar_allreduce), one cudaMemcpyAsync per rank
 * back into h_out[r].  Returns after enqueueing; the caller synchronises
 * `stream` before reading h_out.  AR_ERR_INVALID_ARG if the staging was not
 * reserved or count > max_count.
 * Not capturable: a call on a stream that is being captured into a CUDA
 * graph returns AR_ERR_UNSUPPORTED and enqueues nothing (the device pointer
 * table is copied from memory that lives only for the duration of the call,
 * and pageable copies cannot be captured).  Capture ar_allreduce on device
 * buffers instead.
 */
ar_status_t ar_reserve_host_staging(ar_handle_t h);
ar_status_t ar_allreduce_host(ar_handle_t h, const void* const* h_in,
                              void* const* h_out, size_t count, void* stream);

/* ---- test hooks (faults made on the host side) --------------------------
 *
 * ar_debug_skip_producer -- for the NEXT call of a packet variant only
 * (AR_FUSED_LL8, AR_FUSED_LL8_STAGED, AR_PACKET_3OP), virtual rank `rank`
 * stores none of its scatter packets, so every owner's wait for that rank
 * runs out after the spin limit, the error word is set and ar_last_timeout
 * names `rank` as the missing one.  -1 clears.
 * No memory is touched out of bounds and no wait is unbounded.
 *
 * ar_debug_set_epoch / ar_debug_get_epoch -- synchronous write / read of
 * the device epoch (for testing the wrap from 2^32-1 to 1, which skips 0).
 * Setting it also zeroes every packet region (and writes the zeros back to
 * memory), so that no packet left from before the jump can match the new
 * epoch's flags (in normal use the epoch only moves forward one step per
 * call, and a stale match needs a full 2^32 wrap).
 */
ar_status_t ar_debug_skip_producer(ar_handle_t h, int rank);

/* ar_debug_check_guards -- synchronise the device, then check the guard
 * zones (4 KiB of a fixed byte value before and after each packet region the
 * handle owns: the scatter scratch, the result scratch and the rings), which
 * nothing in the library writes.  *intact = 1 if every guard byte still holds
 * its value, 0 if some kernel wrote outside a packet region.  AR_ERR_CUDA if
 * a copy fails, AR_ERR_INVALID_ARG for a NULL argument.  A stand-in for a
 * memory checker on the library's own buffers (output buffers belong to the
 * caller, who can surround them with guards of its own). */
ar_status_t ar_debug_check_guards(ar_handle_t h, int* intact);

/* ar_debug_delay_producer -- for every later AR_FUSED_LL8 or
 * AR_FUSED_LL8_STAGED call (until cleared with rank -1 or ns 0), the warps of
 * virtual rank `rank` wait `ns` nanoseconds of the device's global timer
 * before their first packet store,
 * so every owner polls for that rank's packets longer than the others'.
 * This is the skewed producer of "Add HIP-graph capture coverage for the
 * sharded-relay collectives" (meta-pytorch/torchcomms #3850, summary:
 * replays with some ranks delayed so that a stale flag or stale staging
 * fails deterministically), made on one GPU.  The value is taken at launch,
 * so a captured call keeps it on every replay.  The wait is bounded (ns <=
 * 10 ms, AR_ERR_INVALID_ARG above) and shorter than any spin limit a test
 * sets, so no wait runs out because of it. */
ar_status_t ar_debug_delay_producer(ar_handle_t h, int rank, uint64_t ns);
ar_status_t ar_debug_set_epoch(ar_handle_t h, uint32_t epoch);
ar_status_t ar_debug_get_epoch(ar_handle_t h, uint32_t* epoch);

/* ---- allocation-free entry point ----------------------------------------
 *
 * The pages have no counterpart to this call; it exists for callers of this
 * library that cannot allocate device memory themselves, so cannot use
 * ar_create: for example a plugin running inside a host framework whose
 * allocator has already reserved the device memory budget and forbids side
 * allocations, or a process that must not allocate once it has started
 * serving.
 *
 * ar_allreduce_fused_noalloc -- the AR_FUSED_LL8 allreduce of bf16 buffers
 * (R <= AR_MAX_PACKET_RANKS) without a handle.
 * Same arguments and result as ar_allreduce (R = rank count,
 * 1..AR_MAX_PACKET_RANKS; device pointer tables; count elements per rank;
 * stream), but the packet
 * scratch and the epoch/counter/error block live in fixed arrays inside the
 * library's device image (AR_NOALLOC_SCRATCH_BYTES of scratch plus 64 bytes),
 * which every GPU that loads the library holds until the process exits.  It
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *   - The first call on each device sets that device up, synchronously:
 *     it looks up the arrays' device addresses, zeroes the scratch and
 *     starts the epoch at 1.  Make that first call before any stream capture.
 *   - count must be <= AR_NOALLOC_MAX_COUNT(R) (about 1.19 M elements for
 *     R = 8, 8.4 M for R = 2, no limit for R = 1); a larger count returns
 *     AR_ERR_INVALID_ARG and launches nothing.  count = 0 returns AR_OK.
 *   - Every call on a device shares the one array and the one epoch, which
 *     keep the last call's contents; the kernel needs nothing cleared between
 *     calls (stale packets carry older epochs, the done counter is left at 0
 *     by the call before).  Calls that overlap on the GPU (other streams, or
 *     other threads) race on the array and give wrong results: order them.
 *   - A packet wait that gives up (100 ms) is recorded in the device-side
 *     error word, which no entry point reads back for this call; that call's
 *     outputs are then undefined.
 * Errors: AR_ERR_INVALID_ARG (R < 1 or R > AR_MAX_PACKET_RANKS, NULL table,
 * count too large), AR_ERR_UNSUPPORTED (device ordinal >= 64), AR_ERR_CUDA
 * (set-up or launch).
 */
#define AR_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
#define AR_NOALLOC_MAX_COUNT(R)                                                   \
  ((R) <= 1 ? (size_t)-1                                                          \
            : (AR_NOALLOC_SCRATCH_BYTES / ((size_t)32 * (size_t)(R) * (size_t)((R)-1))) * \
                  (size_t)8 * (size_t)(R))
ar_status_t ar_allreduce_fused_noalloc(int R, const void* const* d_in_tbl,
                                       void* const* d_out_tbl, size_t count, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* AR_GB300_H */
