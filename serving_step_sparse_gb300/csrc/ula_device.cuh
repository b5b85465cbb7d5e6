// Device-side layout of the KV residency context and the kernel parameter
// blocks.  Shared by the kernels (ula_kernels.cu) and the host orchestrator
// (ula_api.cu); not part of the public ABI (include/ula.h is).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "ula.h"

namespace ula {

constexpr uint32_t kPad = ULA_ADDR_PAD;
constexpr uint32_t kUnalloc = ULA_MAP_UNALLOCATED;
constexpr uint32_t kHostBit = ULA_MAP_HOST;
constexpr uint32_t kSlotMask = 0x7FFFFFFFu;
constexpr uint32_t kNone = 0xFFFFFFFFu;     // no owner / free stamp
constexpr uint32_t kHostPos = 0xFFFFFFFFu;  // work entry on the host-free bitmap
constexpr uint32_t kSegBits = 1024;         // slots per segment (one level-1 word)

// A bitmap with two summary levels.  Level 0: one bit per slot.  Level 1: bit
// i is set iff level-0 word i is nonzero.  Level 2: bit i is set iff level-1
// word i is nonzero.  A level-1 word covers a "segment" of 1,024 slots, a
// level-2 word a "superblock" of 32,768 slots.  Beside the bitmap, `cnt`
// holds the number of set bits of every segment, kept exact by the same
// atomics that flip the bits; victim selection walks these counts in class
// order and stops as soon as the quota is reached.
struct Dims {
  uint32_t n0, n1, n2;
};

struct Bitmap {
  uint32_t *w0, *w1, *w2;
  uint32_t *cnt;  // [n1] set bits per segment
};

__host__ __device__ inline Dims dims_for(uint32_t nbits) {
  Dims d;
  d.n0 = (nbits + 31) / 32;
  d.n1 = (d.n0 + 31) / 32;
  d.n2 = (d.n1 + 31) / 32;
  return d;
}

// Per-group counters living in device memory.
struct GroupCounters {
  uint32_t free_gpu;   // free GPU slots
  uint32_t free_host;  // free host slots
  uint32_t U, M, hits; // last step: unique addresses, misses, hits
  uint32_t F;          // last step: victims taken from free slots (alloc: GPU placements)
  uint32_t K;          // last step: write-backs (alloc: host placements)
  uint32_t Mx;         // last step: misses gathered from the host pool in place (bypass)
  uint32_t n_work;     // selection work entries (GPU classes, then host)
  uint32_t n_work_gpu; // of which on GPU-slot classes
  uint32_t done[3];    // "last block" tickets of the multi-block kernels
  uint32_t lru_lo;     // exact LRU: a lower bound of every occupied slot's stamp
  unsigned long long stat[13];  // ula_stats order
};

enum StatIdx {
  kStSteps = 0, kStEntries, kStUniq, kStHits, kStMisses, kStVictFree, kStVictCold,
  kStVictRing, kStWriteback, kStRows, kStBytesH2D, kStBytesD2H, kStBypassed, kStCount
};

// Everything one group owns on the device.
struct GroupDev {
  uint32_t *map;       // [max_logical]: kUnalloc | GPU slot | kHostBit|host slot
  uint32_t *owner;     // [S]: logical address in the slot or kNone
  uint32_t *stamp;     // [S]: round of last access (defines the bucket), kNone if free
  uint32_t *cls0;      // [B+2][n0]: ring buckets 0..B-1, cold (B), free (B+1)
  uint32_t *cls1;      // [B+2][n1]
  uint32_t *cls2;      // [B+2][n2]
  uint32_t *clsc;      // [B+2][n1]: set bits per segment
  uint32_t *hf0, *hf1, *hf2, *hfc;  // host-free bitmap levels and segment counts
  uint8_t *gpu_pool;   // [S][L][W]
  uint8_t *host_pool;  // [H][L][W], pinned host memory (device pointer)
  uint32_t *uniq;      // [max_entries]: this group's unique addresses of its last step
  uint32_t *row_slot;  // [max_entries]: GPU slot of unique row u if it hit, kNone if it missed
  uint32_t *hitbits;   // [n0]: slots hit in this step (PB-LRU marking), cleared by the marking
  uint32_t *victims;   // [decision_cap]: victim i serves miss i (alloc: GPU slots)
  uint32_t *wb_host;   // [decision_cap]: host slot of write-back j (alloc: host slots)
  uint4 *work;         // [(B+1)*nseg + hseg]: (order position, segment, first rank, count)
  GroupCounters *cnt;
  // per-layer signal (ULA_FLAG_LAYER_SIGNAL only; NULL otherwise)
  uint32_t *layer_flag;  // [L]: round whose output of layer j is complete
  uint32_t *layer_cnt;   // [L]: contributions to layer j's signal in this step
  uint32_t *move_done;   // [L + 1]: chunks of layer j moved in this step; [L]: dispenser
  uint32_t *gather_done; // [L]: gather blocks done with layer j in this step
  unsigned long long *layer_ns;  // [L + 1]: globaltimer at each signal; [L]: step start
  uint32_t layers;     // L_g
  uint32_t pad;
};

struct Geometry {
  uint32_t S, H, B, W;   // GPU slots, host slots, ring buckets, row bytes
  uint32_t max_logical;
  uint32_t bypass;       // ULA_FLAG_BYPASS_OVERFLOW set
  uint32_t exact;        // ULA_FLAG_EXACT_LRU set: occupied slots all in class B, no ring
  uint32_t signal;       // ULA_FLAG_LAYER_SIGNAL set: layer-major fill and per-layer flags
  uint32_t cache;        // TP local buffer: misses are fetched from the owner partitions,
                         // evicted copies are dropped (no host pool, no write-back)
  Dims gd, hd;           // bitmap dims for GPU-slot and host-slot bitmaps
  uint32_t nseg, hseg;   // segments (= level-1 words) per bitmap
  uint32_t fill_shift;   // a miss's host slot >> fill_shift = its bucket in the fill order
};

// Device time span of one launch of a copy kernel (diagnostics): the earliest warp
// start and the latest warp end, both kept as minima (the end complemented), so an
// all-ones record is empty and a ring of records is reset with one memset.
struct SpanRec {
  unsigned long long t0;   // min over warps of the start (globaltimer, ns)
  unsigned long long t1n;  // min over warps of ~end
};
constexpr uint32_t kFillBuckets = 2048;  // buckets of the fill order (host-address order)

__host__ __device__ inline Bitmap class_bitmap(const GroupDev &g, const Geometry &geo, uint32_t c) {
  Bitmap b;
  b.w0 = g.cls0 + (size_t)c * geo.gd.n0;
  b.w1 = g.cls1 + (size_t)c * geo.gd.n1;
  b.w2 = g.cls2 + (size_t)c * geo.gd.n2;
  b.cnt = g.clsc + (size_t)c * geo.gd.n1;
  return b;
}

__host__ __device__ inline Bitmap host_free_bitmap(const GroupDev &g) {
  Bitmap b;
  b.w0 = g.hf0;
  b.w1 = g.hf1;
  b.w2 = g.hf2;
  b.cnt = g.hfc;
  return b;
}

// Victim (or free-slot) selection order: classes at positions 0..n_cls-1.
struct Order {
  uint32_t n_cls;
  uint32_t cls[ULA_MAX_BUCKETS + 2];
};

// TP mode: where a local buffer fetches a missing row (cache mode).  Address t
// lives in partition t % P at local id t / P; map[p] and pool[p] are that
// partition's map and GPU pool for the group being stepped.
constexpr uint32_t kMaxParts = 8;
constexpr uint32_t kSrcShift = 29;  // a cache miss's source: partition << 29 | slot
struct TpSource {
  uint32_t P, S;  // partitions, GPU slots per partition
  const uint32_t *map[kMaxParts];
  const uint8_t *pool[kMaxParts];
};

// Parameters of the per-step kernels of one group.
struct StepParams {
  Geometry geo;
  GroupDev grp;
  Order order;              // free, cold, ring oldest -> newest
  const uint32_t *sel;      // [E]
  uint32_t E, QK, n_req;
  uint32_t epoch;           // dedup epoch of this call
  uint32_t round;           // this round's number r (the current bucket is r % B)
  uint32_t cur;             // r % B
  uint32_t out_cap;
  uint32_t emit_blocks;     // blocks of the rotate+emit kernel that emit (the rest rotate)
  int inject;               // host-side fault injection code (0 = none)
  int32_t *entry_row;       // [E]
  int32_t *req_off;         // [n_req + 1]
  unsigned long long *tbl;  // [max_logical]: (epoch << 32) | ~first entry index
  uint32_t *addr_row;       // [max_logical]: unique row of an address this step
  uint2 *blk;               // [blocks]: (first occurrences, misses) per block, then offsets
  uint32_t *miss_list;      // [max_entries]: misses in first-occurrence order
  uint32_t *miss_hs;        // [max_entries]: host slot of miss i
  uint32_t *miss_row;       // [max_entries]: unique row of miss i
  TpSource src;             // cache mode: the owner partitions
  SpanRec *span;            // the step's metadata span (its start), or NULL
  int *status;              // latched device error (0 = none)
};

// Selection emit (step and alloc): work entries -> victims / host slots.
struct EmitParams {
  Geometry geo;
  const GroupDev *groups;   // device array [G]
  uint32_t group0;          // first group (blockIdx.y adds to it)
  Order order;
  uint32_t quota;           // GPU quota (alloc), or 0xFFFFFFFF = the group's M (step)
  const uint32_t *miss_hs;  // step: [M] host slot of miss i (the fill order's keys)
  uint32_t *fill_order;     // step: [M] out: miss indices in host-slot bucket order (or NULL)
  SpanRec *span;            // step: the metadata span (its end), or NULL
  int *status;
};

struct MoveParams {
  Geometry geo;
  GroupDev grp;
  const uint32_t *sel;        // [E] the step's selection (entry rows are written at commit)
  int32_t *entry_row;         // [E]
  const uint32_t *addr_row;   // [max_logical]
  uint32_t E;
  const uint32_t *miss_list;  // [M] addresses
  const uint32_t *miss_hs;    // [M] their host slots
  const uint32_t *miss_row;   // [M] their unique rows
  uint8_t *out;             // [L][out_cap][W]: the missed rows' outputs (NULL: none)
  uint32_t out_cap;
  uint32_t round, cur;
  TpSource src;               // cache mode: the owner partitions' GPU pools
  const uint32_t *fill_order; // [M]: the order in which the fills run (miss indices)
  uint8_t *stage;             // [M - F][L][W]: the rows of victims F.. staged before the move
  uint32_t *vdone;            // [M]: copies done per victim (reset by its commit)
  SpanRec *span;              // this launch's time span, or NULL
  int *status;
};

// Exact-LRU victim scan (one cooperative launch per step).
constexpr int kLruThreads = 512;
constexpr int kLruDigit = 11;                    // bits per radix-select digit
constexpr uint32_t kLruBins = 1u << kLruDigit;
constexpr int kLruSelectPasses = 3;              // 32-bit keys: 11 + 11 + 10 bits
constexpr uint32_t kSortBins = 256;              // 8-bit digits of the stable sort

struct LruScratch {
  uint4 *blk;          // [2][grid]: per block (min stamp, max stamp, candidates), then
                       // (slots below, at the threshold)
  uint32_t *hist;      // [kLruSelectPasses][kLruBins]
  uint32_t *table;     // [kSortBins][grid] digit counts of a sort pass, then [kSortBins] totals
  uint2 *list[2];      // [max_entries]: (stamp - oldest, slot) of the chosen slots
  uint32_t *bar;       // [3]: grid barrier arrivals, generation; totals buffer parity
  // fast path
  uint32_t *rows;      // [grid][kLruBins]: per-block key counts
  uint32_t *totals;    // [2][kLruBins]: the pool's key counts (one buffer per launch parity)
  uint2 *blist;        // [grid][per]: each block's chosen (key, slot), slot order
  uint32_t per;        // slots per block (a multiple of 4)
};

struct LruParams {
  Geometry geo;
  GroupDev grp;
  LruScratch sc;
  uint32_t round;
  int stall;             // test hook: block 0 skips the first grid barrier
  int *status;
};

struct GatherParams {
  Geometry geo;
  GroupDev grp;
  uint8_t *out;             // [L][out_cap][W]
  uint32_t out_cap;
  uint32_t layer;           // the launch gathers layers [layer, layer + nlayers)
  uint32_t nlayers;
  uint32_t signal;          // contributes to the layers' signals (a step's gather)
  uint32_t round;
  SpanRec *span;            // this launch's time span, or NULL
  int *status;
};

struct AllocParams {
  Geometry geo;
  const GroupDev *groups;
  const uint8_t *rows;      // device-accessible
  unsigned long long group_off[ULA_MAX_GROUPS];  // byte offset of group g's rows
  uint32_t row_stride;      // address i of the range is row i * row_stride (TP partitions)
  uint32_t round[ULA_MAX_GROUPS];
  uint32_t group0;          // first group (blockIdx.y adds to it)
  uint32_t base, n;
  int *status;
};

struct FreeParams {
  Geometry geo;
  const GroupDev *groups;
  uint32_t round[ULA_MAX_GROUPS];
  uint32_t group0;          // first group (blockIdx.y adds to it)
  uint32_t base, n;
  int *status;
};

// Launchers (ula_kernels.cu).  Each returns the launch's cudaError_t.
cudaError_t launch_bitmap_fill(Bitmap b, uint32_t nbits, cudaStream_t s);
// step: (1)(2) dedup + translate + capacity check; (3) rotate + compaction;
// (3b)(4) hit marking, entry rows and the victim walk; (4) victim emit
cudaError_t launch_dedup(const StepParams &p, cudaStream_t s);
cudaError_t launch_rotate_emit(const StepParams &p, cudaStream_t s);
cudaError_t launch_mark_select(const StepParams &p, cudaStream_t s);
cudaError_t launch_select_emit(const EmitParams &p, uint32_t n_groups, int blocks, cudaStream_t s);
// alloc: walk of the free class and the host-free bitmap for a quota of n, per group
cudaError_t launch_alloc_select(const EmitParams &p, uint32_t n_groups, cudaStream_t s);
// the rows of the step's victims that hold data, copied to the staging area (HBM)
cudaError_t launch_stage(const MoveParams &p, int blocks, cudaStream_t s);
// copies, then commit; dependent = chained by programmatic dependent launch to the
// previous kernel on s (false when s waits on an event in between)
cudaError_t launch_move(const MoveParams &p, int blocks, bool dependent, cudaStream_t s);
int move_threads();
cudaError_t launch_gather(const GatherParams &p, int blocks, cudaStream_t s);
// exact LRU: victims [F, M) by a scan of the slot timestamps (cooperative launch of
// `blocks` co-resident blocks)
cudaError_t launch_lru_select(const LruParams &p, int blocks, cudaStream_t s);
cudaError_t lru_resident_blocks(int *per_sm);
// TP mode: part_sel[p * stride + e] = the entry as partition p sees it (a local id, or
// a pad if p does not own it), buf_sel[r * stride + e] = the entry if rank r does not own it
cudaError_t launch_tp_split(const uint32_t *sel, uint32_t E, uint32_t P, uint32_t *part_sel,
                            uint32_t *buf_sel, uint32_t stride, cudaStream_t s);
// a model consumer of one layer (diagnostics): waits for the layer's flag, sums the rows
cudaError_t launch_consume(const uint32_t *flag, uint32_t round, const uint8_t *out,
                           uint32_t out_cap, uint32_t layer, uint32_t n_rows, uint32_t W,
                           unsigned long long *result, cudaStream_t s);
cudaError_t launch_alloc_place(const AllocParams &p, uint32_t n_groups, int max_blocks,
                               cudaStream_t s);
cudaError_t launch_free(const FreeParams &p, uint32_t n_groups, cudaStream_t s);
// blocks of the move and of the hit gather (for rows of up to slot_bytes) that fit on an SM
cudaError_t resident_blocks(int *move_per_sm, int *gather_per_sm, uint32_t slot_bytes);

}  // namespace ula
