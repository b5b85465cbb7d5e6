/*
 * ula.h -- C ABI of the per-decode-step KV residency path for index-based
 * sparse attention, single-GPU DP mode (one HBM slot pool plus one pinned
 * host slot pool per layer group form one logical address space).
 *
 * Source of the operations: "UlaCache: Unified Logical Addressing for Sparse
 * LLM Serving" (paper summary page):
 *   §2 "Unified logical addresses" -- the engine allocates and selects KV by
 *      logical address only; a mapping table names the GPU slot or CPU slot
 *      holding each entry; in DP mode a GPU owns its GPU pool and CPU pool and
 *      an entry lives in exactly one of them; a layer group sharing one
 *      sparse selection does address lookup and dedup once and prefetches
 *      later layers on a separate CUDA stream.
 *   §3 "PB-LRU" -- bucketed replacement for the shared GPU pool: one bucket
 *      per scheduling round, a ring of buckets plus a cold bucket per layer
 *      group, rotation/fold by relabelling, victims from free slots, then
 *      cold, then ring oldest to newest, never the current bucket; bitmaps
 *      with summary levels; data moves first, then the map, then a signal.
 *
 * Conventions for every call:
 *   - Pointers are plain pointers.  "device" = CUDA device memory of the
 *     context's device; "host" = host memory; "device-accessible" = device
 *     memory or pinned (page-locked) host memory.
 *   - Streams and events are cudaStream_t / cudaEvent_t passed as void*.
 *   - Every call returns ULA_OK or an error code.  Errors the host can see
 *     (bad arguments, capacity known on the host) return at once and change
 *     nothing.  Errors only the device can see (an unmapped selected address,
 *     a step needing more GPU slots than are evictable) are latched on the
 *     device, the step's remaining kernels do nothing, and the code is
 *     returned by the next ula_sync; from then on the context is poisoned and
 *     every call except ula_destroy returns ULA_ERR_POISONED.
 *   - A context is used from one host thread at a time.
 */
#ifndef ULA_H
#define ULA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ULA_MAX_GROUPS 64
#define ULA_MAX_BUCKETS 64
#define ULA_ADDR_PAD 0xFFFFFFFFu /* a selection entry that selects nothing */

enum {
  ULA_OK = 0,
  ULA_ERR_INVALID_ARG = 1, /* bad argument; nothing changed */
  ULA_ERR_CAPACITY = 2,    /* pools, logical space or output buffer too small */
  ULA_ERR_UNMAPPED = 3,    /* a selected address is out of range or not allocated */
  ULA_ERR_CUDA = 4,        /* a CUDA runtime call failed */
  ULA_ERR_TIMEOUT = 5,     /* a bounded device wait expired */
  ULA_ERR_POISONED = 6,    /* an earlier device-side error poisoned the context */
  ULA_ERR_INTERNAL = 7     /* a device-side consistency check failed */
};

typedef struct ula_ctx ula_ctx;

typedef struct ula_config {
  uint32_t row_bytes;        /* bytes of one KV row of one layer; multiple of 16 (656 for an
                                FP8 MLA row: 512 e4m3 + 4 fp32 scales + 64 bf16 rope) */
  uint32_t n_groups;         /* G: layer groups, each sharing one selection (1..ULA_MAX_GROUPS) */
  uint32_t layers_per_group[ULA_MAX_GROUPS]; /* L_g >= 1 for g < n_groups */
  uint32_t gpu_slots;        /* S: GPU slots per group (1 .. 2^31-1) */
  uint32_t host_slots;       /* H: host slots per group (0 .. 2^31-1) */
  uint32_t ring_buckets;     /* B: ring buckets per group, including the current one (1..64) */
  uint32_t max_logical;      /* logical addresses live in [0, max_logical) (1 .. 2^31-1) */
  uint32_t max_entries;      /* largest n_req*q*k of one ula_step_group call */
  uint32_t flags;            /* ULA_FLAG_* below; other bits must be 0 */
} ula_config;

/* Overflow bypass (an extension; the pages have no counterpart).  Without it, a step
 * whose misses cannot all be made resident fails with ULA_ERR_CAPACITY.  With it, the
 * first M' = min(misses, S - hits, free GPU + free host slots) misses (in dedup order)
 * are moved as usual and every later miss is gathered straight from its host slot into
 * the output: it stays on the host and nothing else changes for it. */
#define ULA_FLAG_BYPASS_OVERFLOW 1u

/* Exact LRU in place of PB-LRU: the baseline replacement policy that §3 "PB-LRU" sets
 * PB-LRU against (a timestamp per slot, victims found by scanning the whole pool).
 * Every GPU slot keeps the round of its last access (a hit, a fill, or an alloc
 * placement, which counts in the latest round); victims are the free slots, lowest
 * first, then the occupied slots in ascending (timestamp, slot) order, found by a
 * scan of all S timestamps (a radix select of the oldest, then a stable sort of the
 * chosen ones).  A slot accessed in the current round is never chosen.  There are no
 * ring buckets: every occupied slot carries the cold label (diagnostics), and the
 * victims_cold counter counts the occupied slots taken.  Pairing, write-back slots,
 * capacity, the bypass and the move -> map -> signal order are as for PB-LRU.  The
 * scan runs as one cooperative launch whose grid-wide barriers are bounded waits: a
 * wait that expires latches ULA_ERR_TIMEOUT. */
#define ULA_FLAG_EXACT_LRU 2u

/* Per-layer signal (§2, the paragraph on layer groups sharing a selection: a layer
 * computes while later layers' data arrives; §3: data first, then the signal).  The fill runs layer by
 * layer (layer 0 of every miss, then layer 1, ...), and as soon as out[j] holds every
 * unique row of the step (hit rows gathered, missed rows filled) the library stores
 * the step's round number into the group's device flag j (a release store).  A
 * consumer kernel on any stream may then start on layer j while later layers are
 * still moving: it polls the flag with acquire loads until it equals the round that
 * ula_layer_signal reports, with a bound of its own.  layer_ready events are still
 * recorded.  The map commit follows the last layer, as without the flag. */
#define ULA_FLAG_LAYER_SIGNAL 4u

/* The hit gather beside the move.  By default a step gathers its hit rows after its
 * metadata and starts the move (write-back and fill) when the gather is done: the move's host-link traffic and the gather's HBM traffic slow each other
 * down on the SMs they share (the gather ran at about a third of its rate beside the
 * move, on a GB300), so the step keeps them apart.  With this flag the gather runs
 * on a low-priority stream beside the move instead: the step's outputs are complete
 * sooner when the host link is the bottleneck, at the price of every HBM-bound kernel
 * that runs beside the move (this gather, or the caller's attention) going slower.
 * ULA_FLAG_LAYER_SIGNAL implies it. */
#define ULA_FLAG_GATHER_BESIDE_MOVE 8u

/* ULA_FLAG_LAYER_SIGNAL: *d_flags receives the device address of group `group`'s
 * flags (uint32 [L_g], owned by the context, valid until ula_destroy); *round receives
 * the round number of the group's most recently issued ula_step_group (rounds count
 * from 1; 0 before the first step).  Layer j of that step's output is complete once
 * flag j equals *round.  INVALID_ARG without the flag or for a bad group. */
int ula_layer_signal(ula_ctx *ctx, uint32_t group, const uint32_t **d_flags, uint32_t *round);

/* Counters accumulated since ula_create, summed over groups. */
typedef struct ula_stats {
  uint64_t steps;          /* ula_step_group calls completed */
  uint64_t entries;        /* selection entries (pads included) */
  uint64_t uniq;           /* distinct addresses after dedup */
  uint64_t hits;           /* distinct addresses found on the GPU */
  uint64_t misses;         /* distinct addresses filled from the host pool */
  uint64_t victims_free;   /* victims taken from free slots */
  uint64_t victims_cold;   /* victims taken from the cold bucket */
  uint64_t victims_ring;   /* victims taken from ring buckets */
  uint64_t writebacks;     /* victims that held data and were written back */
  uint64_t rows_gathered;  /* (address, layer) rows written to gather outputs */
  uint64_t bytes_h2d;      /* fill (and bypass) bytes moved host -> GPU */
  uint64_t bytes_d2h;      /* write-back bytes moved GPU -> host */
  uint64_t bypassed;       /* misses gathered from the host pool in place (overflow bypass) */
} ula_stats;

/*
 * ula_create -- set up one residency context over caller-owned pools (§2, DP mode).
 *   cfg        : host; copied.
 *   gpu_pools  : host array [G] of device pointers; pool g is [S][L_g][row_bytes] bytes,
 *                16-byte aligned, owned by the caller, borrowed until ula_destroy.
 *   host_pools : host array [G] of pinned host pointers (cudaHostAlloc / pinned tensors);
 *                pool g is [H][L_g][row_bytes]; may be NULL when H == 0.  Borrowed.
 *   stream     : the context's home stream: alloc/free are ordered after the work already
 *                on it, and it waits for them; NULL = legacy stream.
 *   out        : receives the context.
 * The library allocates its metadata (map, slot stamps, bitmaps, scratch, and a
 * staging area of min(max_entries, S) slots of the largest group for the write-backs)
 * with cudaMalloc here and frees it in ula_destroy; it creates three internal streams
 * (the step's critical path and the hit gather's two placements).
 * All slots start free; the current ring bucket starts at 0.
 */
int ula_create(const ula_config *cfg, void *const *gpu_pools, void *const *host_pools,
               void *stream, ula_ctx **out);

/*
 * ula_alloc -- allocate n new logical addresses [*logical_base, *logical_base + n) (§2).
 * Bases are handed out monotonically and never reused.  For each group, each new
 * address takes the lowest free GPU slot (and joins the current ring bucket, as
 * an access in the latest round) or, when none is free, the lowest free host slot,
 * in address order.  Alloc never evicts.
 *   rows : device-accessible; for each group in order, [n][L_g][row_bytes] bytes
 *          (groups concatenated); copied into the chosen slots.  Must stay valid
 *          until the work completes on the home stream (e.g. ula_sync).
 * Errors (host-detected, nothing changed): INVALID_ARG (rows not device-accessible),
 * CAPACITY (n exceeds free slots of both tiers, or the logical space).
 * Asynchronous on the home stream.
 */
int ula_alloc(ula_ctx *ctx, uint32_t n, const void *rows, uint32_t *logical_base);

/*
 * ula_free -- release logical addresses [logical_base, logical_base + n) in every
 * group: their GPU slots become free (leaving their bucket), their host slots free.
 * Errors (host-detected, nothing changed): INVALID_ARG if any address is not live.
 * Asynchronous on the home stream.
 */
int ula_free(ula_ctx *ctx, uint32_t logical_base, uint32_t n);

/*
 * ula_step_group -- one scheduling round of group g for one decode step (§2, §3).
 * In stream order, all on the device:
 *   (1) dedup the selection (first occurrences in flattened (request, query, i) order),
 *   (2) translate through the map (GPU slot = hit, host slot = miss),
 *   (3) rotate the ring (the current bucket advances; the reused bucket's slots fold
 *       into cold -- labels only) and move every hit into the current bucket,
 *   (4) pick one victim per miss through the summary bitmaps: free slots, then cold,
 *       then ring buckets oldest to newest, never the current bucket, lowest slot
 *       first; victim i serves miss i,
 *   (5) write each victim that holds data back to the host pool (the j-th such victim
 *       to the j-th lowest free host slot), fill each miss from its host slot, then
 *       update the map (moves complete before the map changes) and signal,
 *   (6) gather out[j][u] = layer j of unique address u, for every layer of the group.
 *       Rows that hit are gathered, every layer in one launch (their slots never move
 *       in this round): by default after the step's metadata and before the move, on
 *       the context's copy stream; with ULA_FLAG_GATHER_BESIDE_MOVE on an internal
 *       low-priority stream as soon as the compaction has recorded their slots, beside
 *       the marking, the victim choice and the move.  The gather moves whole rows with
 *       bulk copies through shared memory (blocks of 16 threads, one row buffer each:
 *       42 KB per block for 4 layers of 656 bytes; rows longer than 6,392 bytes go
 *       through registers instead).  Rows that missed are written by the fill itself,
 *       from the bytes it moves.
 * The move writes every victim that holds data back from a staging copy in HBM (made
 * right after the victims are known), so its write-backs (in victim order, which is
 * ascending host-slot order) and its fills (sorted by the miss's host slot) each
 * sweep the host pool in address order; the pairing of miss i with victim i is
 * unchanged.
 * The work runs on the context's internal highest-priority stream, ordered after
 * everything already enqueued on `stream`; `stream` is made to wait for the commit
 * and for the hit gather, so work the caller enqueues next on `stream` sees every
 * output; layer_ready events are recorded at that point too.
 *   d_sel       : device [n_req][q][k] uint32 logical addresses; ULA_ADDR_PAD = none.
 *   d_out       : device [L_g][out_cap_rows][row_bytes]; rows [0, U) are written.
 *   d_entry_row : device [n_req*q*k] int32: row u of each entry, -1 for pads.
 *   d_req_off   : device [n_req+1] int32: unique rows first seen in request r are
 *                 [req_off[r], req_off[r+1]); req_off[n_req] = U.
 *   layer_ready : host array [L_g] of cudaEvent_t recorded when layer j of d_out is
 *                 ready (on the stream that wrote it), or NULL.
 *   stream      : the caller's stream; the step is ordered after every earlier call on
 *                 this context.  Returns without waiting for the device.
 * Device-detected errors (latched, returned by ula_sync, nothing changed by the step):
 * UNMAPPED (an address >= max_logical or not allocated), CAPACITY (misses > S - hits or
 * write-backs > free host slots, unless ULA_FLAG_BYPASS_OVERFLOW; or U > out_cap_rows).
 * Host-detected: INVALID_ARG (group out of range, n_req*q*k > max_entries, NULL buffers).
 */
int ula_step_group(ula_ctx *ctx, uint32_t group, const uint32_t *d_sel, uint32_t n_req,
                   uint32_t q, uint32_t k, void *d_out, uint32_t out_cap_rows,
                   int32_t *d_entry_row, int32_t *d_req_off, void *const *layer_ready,
                   void *stream);

/*
 * ula_sync -- wait for all work of the context (all its streams), then return the first
 * latched device error (or ULA_OK).  stats: host, optional; receives the counters.
 */
int ula_sync(ula_ctx *ctx, ula_stats *stats);

/* ula_destroy -- wait for the context's work and free everything it allocated. */
void ula_destroy(ula_ctx *ctx);

/* Text for an error code (static storage). */
const char *ula_error_string(int code);

/* ------------------------------------------------------------ diagnostics
 * For tests and tools: sizes of the internal arrays, a blocking copy of one group's
 * state, and host-side fault injection.  Bitmap words are 32-bit, bit b of word w is
 * slot 32*w + b; level 1 holds one bit per level-0 word (set iff that word is
 * nonzero), level 2 one bit per level-1 word.  Classes: 0..B-1 ring buckets, B cold,
 * B+1 free.  Map entries: ULA_MAP_UNALLOCATED, a GPU slot, or ULA_MAP_HOST | host slot.
 */
#define ULA_MAP_UNALLOCATED 0xFFFFFFFFu
#define ULA_MAP_HOST 0x80000000u
#define ULA_STAMP_FREE 0xFFFFFFFFu

typedef struct ula_debug_layout {
  uint32_t n0, n1, n2;   /* words per level of a GPU-slot bitmap */
  uint32_t h0, h1, h2;   /* words per level of the host-free bitmap */
  uint32_t n_classes;    /* B + 2 */
  uint32_t decision_cap; /* capacity of the victim / write-back lists */
} ula_debug_layout;

typedef struct ula_debug_state {
  /* host buffers to fill; NULL skips */
  uint32_t *map;            /* [max_logical] */
  uint32_t *owner;          /* [S] logical address in each GPU slot, 0xFFFFFFFF if none */
  uint32_t *stamp;          /* [S] round of last access, ULA_STAMP_FREE if free */
  uint32_t *class_bits;     /* [n_classes][n0] */
  uint32_t *class_sum1;     /* [n_classes][n1] */
  uint32_t *class_sum2;     /* [n_classes][n2] */
  uint32_t *host_free_bits; /* [h0] */
  uint32_t *host_free_sum1; /* [h1] */
  uint32_t *host_free_sum2; /* [h2] */
  uint32_t *uniq;           /* [max_entries]: last step's unique addresses */
  uint32_t *victims;        /* [decision_cap]: last step's victims (first M) */
  uint32_t *wb_host;        /* [decision_cap]: last step's write-back host slots (first K) */
  uint32_t *class_seg_count;/* [n_classes][n1]: set bits per 1,024-slot segment */
  uint32_t *host_seg_count; /* [h1] */
  uint32_t *row_slot;       /* [max_entries]: GPU slot of each unique row after the commit */
  /* filled always */
  uint32_t round;           /* rounds completed by this group */
  uint32_t cur;             /* current ring bucket = round % B */
  uint32_t free_gpu, free_host;
  uint32_t U, M, hits, victims_free, writebacks; /* last step */
} ula_debug_state;

int ula_debug_layout_get(const ula_ctx *ctx, ula_debug_layout *out);
int ula_debug_export(ula_ctx *ctx, uint32_t group, ula_debug_state *st);
/* The next ula_step_group latches `code` on the device before it changes anything
 * (host-side fault injection for tests of the error path; no GPU fault).  With
 * code ULA_DEBUG_STALL_SCAN_BARRIER instead, in the next step's exact-LRU scan one
 * block never arrives at the first grid-wide barrier: the other blocks wait out
 * their bound (about one second), latch ULA_ERR_TIMEOUT and return (a test of the
 * bounded wait; nothing hangs). */
int ula_debug_inject(ula_ctx *ctx, int code);
#define ULA_DEBUG_STALL_SCAN_BARRIER 0x100
/* ULA_FLAG_LAYER_SIGNAL: waits for the context's work (like ula_sync, without its
 * error check), then copies group `group`'s signal times into ns (host, [L_g + 1]):
 * ns[j] = device globaltimer (ns) when layer j's flag was set in the last step,
 * ns[L_g] = when that step started.  For measuring how early each layer is ready. */
int ula_debug_layer_times(ula_ctx *ctx, uint32_t group, unsigned long long *ns);
/* ULA_FLAG_LAYER_SIGNAL: a model consumer of one layer.  Launches at once on `stream`
 * one block that polls group `group`'s flag `layer` with acquire loads until it equals
 * `round` (bounded: 1 s), then reads out[layer][0, n_rows) (d_out as given to the step,
 * [L_g][out_cap_rows][row_bytes]) and writes into d_result (device, u64 [3]): the
 * globaltimer when it saw the flag, the wrapping sum of the rows' 32-bit words, and a
 * status (0, or ULA_ERR_TIMEOUT when the bound expired).  It changes no state; it
 * shows what a consumer on another stream does while later layers are still moving. */
int ula_debug_consume(ula_ctx *ctx, uint32_t group, uint32_t layer, uint32_t round,
                      const void *d_out, uint32_t out_cap_rows, uint32_t n_rows,
                      unsigned long long *d_result, void *stream);
/* Re-run the gather of the hit rows of `group`'s last step for layers
 * [layer, layer + n_layers) in one launch (the step gathers all layers in one), into d_out ([L_g][out_cap_rows][row_bytes], device) on `stream`,
 * changing no state (for timing the gather kernel on its own).  Launches at once: the
 * caller orders it after the step (e.g. ula_sync) and before the group's slots change
 * again (its next step, or any alloc/free).  n_layers 0 or past L_g is
 * ULA_ERR_INVALID_ARG; more rows than out_cap_rows latch ULA_ERR_CAPACITY. */
int ula_debug_regather(ula_ctx *ctx, uint32_t group, uint32_t layer, uint32_t n_layers,
                       void *d_out, uint32_t out_cap_rows, uint32_t blocks_per_sm,
                       void *stream);
/* blocks_per_sm: 0 = the grid the step uses; otherwise that many blocks per SM (at most
 * what fits). */

/* ------------------------------------------------------------ profiling
 * Kernel launches are counted per phase always.  When enabled, every phase
 * instance is bracketed by two CUDA events recorded on the stream it is launched
 * on, and ula_profile_read sums their durations.  Reading synchronises the context.
 */
enum {
  ULA_PHASE_DEDUP = 0,  /* dedup, translate, capacity check */
  ULA_PHASE_ROTATE,     /* ring rotation + compaction of unique rows and misses */
  ULA_PHASE_MARK,       /* hit marking, entry rows, victim walk over segment counts */
  ULA_PHASE_SELECT,     /* victim (or free-slot) index emission, the fill order */
  ULA_PHASE_MOVE,       /* write-back, fill (and the missed rows' outputs), map commit */
  ULA_PHASE_GATHER,     /* the gather of the hit rows (every layer in one launch) */
  ULA_PHASE_ALLOC,      /* alloc placement and copy-in */
  ULA_PHASE_FREE,       /* free */
  ULA_PHASE_STAGE,      /* victims' rows copied to the staging area before the move */
  ULA_PHASE_COUNT
};

typedef struct ula_profile {
  uint64_t kernels[ULA_PHASE_COUNT]; /* kernel launches */
  uint64_t timed[ULA_PHASE_COUNT];   /* phase instances timed (profiling enabled) */
  double ms[ULA_PHASE_COUNT];        /* summed event-timed durations, milliseconds */
} ula_profile;

int ula_profile_enable(ula_ctx *ctx, int on);
/* Copies the accumulated profile into *out (may be NULL) and, if reset != 0, zeroes it. */
int ula_profile_read(ula_ctx *ctx, ula_profile *out, int reset);

/* Launch spans of a step's kernels, measured on the device itself: while recording is
 * on, every launch of the hit gather, the staging copy and the move, and every step's
 * metadata kernels taken together, keep the device globaltimer of the first warp's
 * start and of the last warp's end (two atomics per warp, so recording costs next to
 * nothing and can stay on in a timed run).  Spans of kernels that overlap are kept
 * apart, unlike summed event durations. */
typedef struct ula_span {
  uint32_t phase;     /* ULA_PHASE_GATHER, ULA_PHASE_STAGE, ULA_PHASE_MOVE, or
                         ULA_PHASE_SELECT for the step's metadata: from its first dedup
                         thread to the end of its last victim-emission warp */
  uint32_t group;
  uint64_t start_ns;  /* globaltimer (ns); 0 and 0 when the launch returned early */
  uint64_t end_ns;
} ula_span;
/* Waits for the context's work, clears the recorded spans and turns recording on or
 * off.  At most 65,536 launches are recorded between reads; later ones are not. */
int ula_profile_spans(ula_ctx *ctx, int on);
/* Waits for the context's work, copies the first min(cap, n) of the n spans recorded
 * since the last read or enable (in launch order) into out (host), sets *count = n,
 * and clears them (recording stays as it was). */
int ula_profile_spans_read(ula_ctx *ctx, ula_span *out, uint32_t cap, uint32_t *count);

/* ------------------------------------------------------------ no-allocation dedup
 * The pages have no counterpart for this entry point; it serves callers that must
 * not allocate device memory where they dedup: an engine that reserved nearly all
 * HBM for its KV pools at start-up (a cudaMalloc would fail or fragment the pool),
 * or a latency-critical path that cannot take cudaMalloc's implicit device
 * synchronisation.  It computes the same dedup as ula_step_group's first step,
 * without a context and without allocating: its scratch is a fixed array of about
 * 1.3 MB inside this library, resident on every device that loads the library
 * until the process exits.
 *   d_sel       : device [n] uint32 addresses; ULA_ADDR_PAD entries select nothing.
 *   d_uniq      : device [n] out: distinct addresses in order of first occurrence.
 *   d_entry_row : device [n] out: index into d_uniq of each entry's address, -1 for pads.
 *   d_n_uniq    : device [1] out: number of distinct addresses.
 *   stream      : cudaStream_t (void*); the call is asynchronous on it.
 * n above ULA_NOALLOC_MAX_ENTRIES returns ULA_ERR_CAPACITY; NULL buffers return
 * ULA_ERR_INVALID_ARG (nothing is launched in either case).  The first call on a
 * device looks up the scratch array's device address (with that device current);
 * make that first call before any stream capture.  The address is kept for the life
 * of the process: after a cudaDeviceReset the library's device code may be loaded
 * elsewhere, so the entry point must not be called again in that process.  Every call on a device uses the
 * same scratch and clears what it needs first, so calls that overlap on the GPU
 * (on different streams, or from different host threads) race and must not be
 * issued; calls on one stream are ordered and safe.
 */
#define ULA_NOALLOC_MAX_ENTRIES 65536u
int ula_dedup_noalloc(const uint32_t *d_sel, uint32_t n, uint32_t *d_uniq,
                      int32_t *d_entry_row, uint32_t *d_n_uniq, void *stream);

/*
 * TP mode, emulated on one GPU (§2 "Unified logical addresses", TP paragraph): the
 * pools of P GPUs form one distributed address space in which logical address t
 * lives on "GPU" t mod P, and a GPU that computes caches copies of the entries it
 * fetched from the others.  Here P partitions of this GPU stand in for the P
 * GPUs: partition p is a DP residency context (everything above) over local ids
 * t / P with its own GPU and host pools, and rank r's local buffer (per group) holds
 * copies of remote rows (t mod P != r) in buffer_slots slots under PB-LRU, evicted
 * copies dropped (the owner keeps the entry); a missing row is fetched from its
 * owner partition's GPU slot, where the owner's step has just made it resident (the
 * cross-GPU copy of TP mode, here a copy inside HBM).  Limits: 1 <= P <= 8; TP with
 * ULA_FLAG_LAYER_SIGNAL or ULA_FLAG_EXACT_LRU is not supported (INVALID_ARG).
 *
 * ula_tp_create -- cfg: per partition (gpu_slots, host_slots per partition; max_logical
 *   and max_entries global).  gpu_pools, host_pools: host arrays [P * G] (partition-
 *   major) of pools as for ula_create; buffer_pools: [P * G] device pools of
 *   [buffer_slots][L_g][row_bytes] (rank-major).  stream: the home stream.  Creates
 *   2P contexts and 2P streams; the pools stay caller-owned.
 * ula_tp_alloc -- rows: per group [n][L_g][row_bytes] for global addresses
 *   [base, base + n), device-accessible; each partition takes its every-P-th rows.
 *   Not atomic across partitions: an error can leave earlier partitions allocated.
 * ula_tp_free -- frees the range in every partition and drops every buffered copy.
 * ula_tp_step_group -- one TP step of `group` for the whole selection d_sel (device
 *   [n_req][q][k], global addresses): partition p runs a DP step on the entries it owns
 *   (others as pads, addresses as local ids), writing d_local_out[p] (rows of its own
 *   addresses, first-occurrence order), d_local_entry_row[p], d_local_req_off[p]; then
 *   rank r's buffer takes the entries it does not own, writing d_remote_out[r],
 *   d_remote_entry_row[r], d_remote_req_off[r] (as for ula_step_group; -1 for pads and
 *   for the other side's entries).  Host arrays of P device pointers each; all outputs
 *   [L_g][out_cap_rows][row_bytes].  The partitions run concurrently on their own
 *   streams, the buffers after all of them; `stream` continues after everything.
 *   Device errors latch in the context that met them and are returned by ula_tp_sync.
 * ula_tp_sync -- waits for every context; stats (optional, host [2P]): partition
 *   p's counters at [p], rank r's buffer counters at [P + r] (bytes_h2d = fetched bytes).
 * ula_tp_context -- the context of partition `index` (kind 0) or of rank `index`'s
 *   buffer (kind 1), for the diagnostics above; owned by the TP object.
 */
typedef struct ula_tp ula_tp;
int ula_tp_create(const ula_config *cfg, uint32_t parts, uint32_t buffer_slots,
                  void *const *gpu_pools, void *const *host_pools, void *const *buffer_pools,
                  void *stream, ula_tp **out);
int ula_tp_alloc(ula_tp *tp, uint32_t n, const void *rows, uint32_t *logical_base);
int ula_tp_free(ula_tp *tp, uint32_t base, uint32_t n);
int ula_tp_step_group(ula_tp *tp, uint32_t group, const uint32_t *d_sel, uint32_t n_req,
                      uint32_t q, uint32_t k, void *const *d_local_out,
                      void *const *d_remote_out, uint32_t out_cap_rows,
                      int32_t *const *d_local_entry_row, int32_t *const *d_local_req_off,
                      int32_t *const *d_remote_entry_row, int32_t *const *d_remote_req_off,
                      void *stream);
int ula_tp_sync(ula_tp *tp, ula_stats *stats);
ula_ctx *ula_tp_context(ula_tp *tp, int kind, uint32_t index);
int ula_tp_destroy(ula_tp *tp);

#ifdef __cplusplus
}
#endif

#endif /* ULA_H */
