// Kernels of the KV residency path (sm_103a).  Integer, bitmap and copy work:
// no tensor cores, nothing here is a contraction.
//
// Source of the method: "UlaCache: Unified Logical Addressing for Sparse LLM
// Serving" (paper summary page), §2 "Unified logical addresses" (map, DP-mode
// exclusive tiers, per-group dedup, side-stream prefetch) and §3 "PB-LRU"
// (bucket ring + cold bucket, rotation by relabelling, victim order, bitmaps
// with summary levels, parallel hit detection/dedup, move -> map -> signal).
//
// One step of one group is five metadata launches, chained by programmatic
// dependent launch:
//   k_dedup_stamp       (1) every entry bids to be its address's first occurrence
//   k_dedup_count_scan  (1)(2) per-block counts of first occurrences / misses; the
//                       last block scans them and runs the capacity check
//   k_rotate_emit       (3a) ring rotation + cold fold (labels only), and the
//                       compaction of unique rows / misses / CSR offsets; each hit's
//                       slot, stamp and bit in the step's hit map
//   k_mark_select       (3b) the hit map applied to the labels, word by word; the last
//                       block walks the segment counts (4) in class order
//   k_select_emit       (4) the victims' and write-back slots' indices; (5) the order
//                       of the fills (one more block)
// then three copy launches, one after the other:
//   k_gather_bulk       (6) every layer of the rows that hit (hit slots never move in
//                       their round), a whole row per bulk copy through shared memory
//                       (k_gather, with registers, for rows too long for its buffers)
//   k_stage             (1) entry rows; (5) the rows of the victims that hold data,
//                       copied to the staging area
//   k_move              (5) write-backs (from the staging area) and fills over the host
//                       link, then each victim's map, labels and host slot; (6) the
//                       missed rows' outputs
// Options: k_lru_select (exact LRU's scan, after the marking), the gather beside the
// move, k_move_layers + k_commit (per-layer signal), cache mode (a TP rank's local
// buffer).
//
// Concurrency discipline for the bitmaps: inside one kernel a given bitmap is
// either only set or only cleared.  That keeps the summary levels and the
// segment counts exact with plain atomics: a set that finds its word empty sets
// the level-1 bit (and so on up), a clear that empties its word clears the
// level-1 bit (and so on up); with only one direction per kernel no set can
// interleave with a clear.
#include "ula_device.cuh"

namespace ula {

namespace {

constexpr int kScanThreads = 1024;
constexpr int kEntryThreads = 1024;  // blocks of the per-entry kernels with block scans
constexpr int kStampThreads = 256;
constexpr int kWalkSegs = 4;        // segments per thread per step of the victim walk
constexpr int kMarkClasses = 8;     // class words a marking warp loads at once

// Launch shapes of the register gather and of the move (build-time tunables).
#ifndef ULA_GATHER_THREADS
#define ULA_GATHER_THREADS 256
#endif
#ifndef ULA_GATHER_MINBLOCKS
#define ULA_GATHER_MINBLOCKS 3
#endif
#ifndef ULA_GATHER_UNROLL
#define ULA_GATHER_UNROLL 12
#endif
#ifndef ULA_MOVE_THREADS
#define ULA_MOVE_THREADS 128
#endif
#ifndef ULA_MOVE_MINBLOCKS
#define ULA_MOVE_MINBLOCKS 4
#endif
#ifndef ULA_MOVE_UNROLL
#define ULA_MOVE_UNROLL 6
#endif
constexpr int kGatherThreads = ULA_GATHER_THREADS;

__device__ __forceinline__ void latch(int *status, int code) { atomicCAS(status, 0, code); }

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may be scheduled before the previous kernel on its stream has
// finished; pdl_wait() returns once that kernel has completed and its writes are
// visible (at once for an ordinary launch), and pdl_launch() lets the next kernel
// be scheduled as soon as every block of this one has issued it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long v;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(v));
  return v;
}

__device__ __forceinline__ void st_release(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// One contribution to layer j's signal (the move's, or the hit gather's): the
// last of `needed` stores the round into the layer's flag, after a fence that
// orders every output write of the contributors before it.
__device__ void layer_contrib(const GroupDev &g, uint32_t j, uint32_t needed, uint32_t round) {
  __threadfence();
  if (atomicAdd(&g.layer_cnt[j], 1u) == needed - 1) {
    g.layer_cnt[j] = 0;
    g.layer_ns[j] = global_ns();
    __threadfence();
    st_release(&g.layer_flag[j], round);
  }
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31; }

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    uint32_t t = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= (uint32_t)d) v += t;
  }
  return v;
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
  for (int d = 16; d; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// Block-uniform early exit on a latched error (safe before __syncthreads).
__device__ __forceinline__ bool block_skips(const int *status) {
  __shared__ int s_status;
  if (threadIdx.x == 0) s_status = *(volatile const int *)status;
  __syncthreads();
  return s_status != 0;
}

// Block-wide inclusive scan of one value per thread (T threads); *total gets the sum.
template <int T>
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, uint32_t *total) {
  __shared__ uint32_t ws[T / 32];
  __shared__ uint32_t tot;
  const uint32_t inc = warp_incl_scan(v);
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  if (lane == 31) ws[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint32_t x = lane < T / 32 ? ws[lane] : 0u;
    const uint32_t y = warp_incl_scan(x);
    if (lane < T / 32) ws[lane] = y;
    if (lane == 31) tot = y;
  }
  __syncthreads();
  const uint32_t r = inc + (warp ? ws[warp - 1] : 0u);
  *total = tot;
  __syncthreads();
  return r;
}

// "Last block done": true in exactly one block, after every block has passed
// this point; that block then sees all other blocks' global writes.
__device__ __forceinline__ bool last_block(uint32_t *ticket) {
  __shared__ bool s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t t = atomicAdd(ticket, 1u);
    s_last = (t == gridDim.x * gridDim.y - 1);
    if (s_last) *ticket = 0;  // ready for the next launch
  }
  __syncthreads();
  if (s_last) __threadfence();
  return s_last;
}

__device__ __forceinline__ void bm_set(Bitmap b, uint32_t bit) {
  const uint32_t i0 = bit >> 5;
  const uint32_t m0 = 1u << (bit & 31);
  const uint32_t old0 = atomicOr(&b.w0[i0], m0);
  if (!(old0 & m0)) atomicAdd(&b.cnt[bit >> 10], 1u);
  if (old0 == 0) {
    const uint32_t i1 = i0 >> 5;
    const uint32_t old1 = atomicOr(&b.w1[i1], 1u << (i0 & 31));
    if (old1 == 0) atomicOr(&b.w2[i1 >> 5], 1u << (i1 & 31));
  }
}

__device__ __forceinline__ void bm_clear(Bitmap b, uint32_t bit) {
  const uint32_t i0 = bit >> 5;
  const uint32_t m0 = 1u << (bit & 31);
  const uint32_t old0 = atomicAnd(&b.w0[i0], ~m0);
  if (old0 & m0) atomicSub(&b.cnt[bit >> 10], 1u);
  if (old0 == m0) {  // this clear emptied the word
    const uint32_t i1 = i0 >> 5;
    const uint32_t m1 = 1u << (i0 & 31);
    const uint32_t old1 = atomicAnd(&b.w1[i1], ~m1);
    if (old1 == m1) atomicAnd(&b.w2[i1 >> 5], ~(1u << (i1 & 31)));
  }
}

// Clear the set bits `mask` of level-0 word i0 at once (clear-only phase).
__device__ __forceinline__ void bm_clear_mask(Bitmap b, uint32_t i0, uint32_t mask) {
  const uint32_t old0 = atomicAnd(&b.w0[i0], ~mask);
  const uint32_t cleared = old0 & mask;
  if (cleared) atomicSub(&b.cnt[i0 >> 5], (uint32_t)__popc(cleared));
  if (old0 && (old0 & ~mask) == 0) {  // this clear emptied the word
    const uint32_t i1 = i0 >> 5;
    const uint32_t m1 = 1u << (i0 & 31);
    const uint32_t old1 = atomicAnd(&b.w1[i1], ~m1);
    if (old1 == m1) atomicAnd(&b.w2[i1 >> 5], ~(1u << (i1 & 31)));
  }
}

// The class of a GPU slot from its stamp: free, cold (last access at least B
// rounds ago: its bucket has been folded), or the ring bucket of its round.
__device__ __forceinline__ uint32_t class_of(uint32_t stamp, uint32_t round, uint32_t B) {
  if (stamp == kNone) return B + 1;
  if (round - stamp >= B) return B;
  return stamp % B;
}

// The class of a slot under the configured policy: exact LRU keeps every
// occupied slot in the one class B (its order lives in the stamps alone).
__device__ __forceinline__ uint32_t slot_class(const Geometry &geo, uint32_t stamp, uint32_t round) {
  if (geo.exact) return stamp == kNone ? geo.B + 1 : geo.B;
  return class_of(stamp, round, geo.B);
}

// The class a slot joins when it is accessed in the round whose bucket is `cur`.
__device__ __forceinline__ uint32_t access_class(const Geometry &geo, uint32_t cur) {
  return geo.exact ? geo.B : cur;
}

// Span of a launch (diagnostics): each warp folds its start and end into the record.
__device__ __forceinline__ void span_open(SpanRec *r) {
  if (r && lane_id() == 0) atomicMin(&r->t0, global_ns());
}
__device__ __forceinline__ void span_close(SpanRec *r) {
  if (r && lane_id() == 0) atomicMin(&r->t1n, ~global_ns());
}

// ------------------------------------------------------------------ init

// all of [0, nbits) set, with exact summaries and segment counts
__global__ void k_bitmap_fill(Bitmap b, uint32_t nbits) {
  const Dims d = dims_for(nbits);
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t w = blockIdx.x * blockDim.x + threadIdx.x; w < d.n0; w += stride) {
    const uint32_t n = nbits - w * 32;
    b.w0[w] = n >= 32 ? 0xffffffffu : ((1u << n) - 1u);
    if (w < d.n1) {
      const uint32_t m = d.n0 - w * 32;
      b.w1[w] = m >= 32 ? 0xffffffffu : ((1u << m) - 1u);
      const uint32_t left = nbits - w * kSegBits;
      b.cnt[w] = left >= kSegBits ? kSegBits : left;
    }
    if (w < d.n2) {
      const uint32_t m = d.n1 - w * 32;
      b.w2[w] = m >= 32 ? 0xffffffffu : ((1u << m) - 1u);
    }
  }
}

// ----------------------------------------------------------------- dedup

__device__ __forceinline__ unsigned long long first_key(uint32_t epoch, uint32_t e) {
  return ((unsigned long long)epoch << 32) | (0xffffffffu - e);
}

// (1) every entry proposes itself as its address's first occurrence; the
// largest key of this epoch = the smallest entry index wins.
__global__ void k_dedup_stamp(StepParams p) {
  pdl_launch();
  if (*(volatile int *)p.status) return;
  const uint32_t e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e == 0 && p.span) atomicMin(&p.span->t0, global_ns());  // the step's metadata starts
  if (p.inject && e == 0) latch(p.status, p.inject);
  if (p.geo.signal && e == 0) p.grp.layer_ns[p.grp.layers] = global_ns();  // step start
  if (e >= p.E) return;
  const uint32_t a = p.sel[e];
  if (a == kPad) return;
  // (a local buffer holds copies: an address it does not hold is a miss, not an error)
  if (a >= p.geo.max_logical || (!p.geo.cache && p.grp.map[a] == kUnalloc)) {
    latch(p.status, ULA_ERR_UNMAPPED);
    return;
  }
  atomicMax(&p.tbl[a], first_key(p.epoch, e));
}

struct Flags {
  uint32_t a, first, miss, m;  // m: the map entry of a first occurrence
};

__device__ __forceinline__ Flags entry_flags(const StepParams &p, uint32_t e) {
  Flags f{kPad, 0, 0, kNone};
  if (e < p.E) {
    f.a = p.sel[e];
    if (f.a != kPad && p.tbl[f.a] == first_key(p.epoch, e)) {
      f.first = 1;
      f.m = p.grp.map[f.a];
      f.miss = (p.geo.cache ? f.m == kUnalloc : (f.m & kHostBit) != 0) ? 1u : 0u;  // (2) translate
    }
  }
  return f;
}

// Per-block counts of first occurrences and misses; the last block turns them
// into exclusive offsets, totals U and M, and runs the capacity check -- no
// state changes before it passes.
__global__ void __launch_bounds__(kEntryThreads) k_dedup_count_scan(StepParams p) {
  pdl_wait();
  pdl_launch();
  if (block_skips(p.status)) return;
  if (p.E == 0 && blockIdx.x == 0 && threadIdx.x == 0) {  // (no entries: no stamp kernel)
    if (p.geo.signal) p.grp.layer_ns[p.grp.layers] = global_ns();  // step start
    if (p.span) atomicMin(&p.span->t0, global_ns());
  }
  const uint32_t e = blockIdx.x * blockDim.x + threadIdx.x;
  const Flags f = entry_flags(p, e);
  __shared__ uint32_t sf[kEntryThreads / 32], sm[kEntryThreads / 32];
  const uint32_t wf = warp_sum(f.first), wm = warp_sum(f.miss);
  if (lane_id() == 0) {
    sf[threadIdx.x >> 5] = wf;
    sm[threadIdx.x >> 5] = wm;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t tf = 0, tm = 0;
    for (int w = 0; w < kEntryThreads / 32; ++w) {
      tf += sf[w];
      tm += sm[w];
    }
    p.blk[blockIdx.x] = make_uint2(tf, tm);
  }
  GroupCounters *c = p.grp.cnt;
  if (!last_block(&c->done[0])) return;
  // the last block: exclusive scan over the block counts
  const uint32_t nblk = gridDim.x;
  uint32_t runf = 0, runm = 0;
  for (uint32_t b0 = 0; b0 < nblk; b0 += kEntryThreads) {
    const uint32_t b = b0 + threadIdx.x;
    const uint2 v = b < nblk ? __ldcg(&p.blk[b]) : make_uint2(0, 0);
    uint32_t totf, totm;
    const uint32_t incf = block_incl_scan<kEntryThreads>(v.x, &totf);
    const uint32_t incm = block_incl_scan<kEntryThreads>(v.y, &totm);
    if (b < nblk) p.blk[b] = make_uint2(runf + incf - v.x, runm + incm - v.y);
    runf += totf;
    runm += totm;
  }
  if (p.E == 0)
    for (uint32_t r = threadIdx.x; r <= p.n_req; r += blockDim.x) p.req_off[r] = 0;
  if (threadIdx.x == 0) {
    const uint32_t U = runf, Mall = runm, hits = U - Mall;
    const uint64_t can_place =
        p.geo.cache ? (uint64_t)p.geo.S - hits  // a buffer drops its victims' copies
                    : min((uint64_t)p.geo.S - hits, (uint64_t)c->free_gpu + c->free_host);
    const uint32_t M = (uint32_t)min((uint64_t)Mall, can_place);  // misses made resident
    const bool ok = U <= p.out_cap && (M == Mall || p.geo.bypass);
    if (!ok) {
      latch(p.status, ULA_ERR_CAPACITY);
    } else {
      c->U = U;
      c->M = M;
      c->Mx = Mall - M;
      c->hits = hits;
      c->F = 0;
      c->K = 0;
      c->n_work = 0;
      c->n_work_gpu = 0;
      if (p.geo.signal) p.grp.move_done[p.grp.layers] = 0;  // the layer-major move's dispenser
      p.req_off[p.n_req] = (int32_t)U;
      const unsigned long long sb = (unsigned long long)p.grp.layers * p.geo.W;
      c->stat[kStSteps] += 1;
      c->stat[kStEntries] += p.E;
      c->stat[kStUniq] += U;
      c->stat[kStHits] += hits;
      c->stat[kStMisses] += Mall;
      c->stat[kStBypassed] += Mall - M;
      c->stat[kStRows] += (unsigned long long)U * p.grp.layers;
      c->stat[kStBytesH2D] += (unsigned long long)Mall * sb;
    }
  }
}

// Blocks [0, emit_blocks): compact first occurrences into uniq (first-occurrence
// order), misses into miss_list (same order), CSR offsets per request, and the
// unique row of every selected address.  Blocks from emit_blocks on: (3a) the
// rotation -- the current bucket advances to `cur` and what is left in it folds
// into the cold bucket (sets on cold, clears on the reused bucket; labels only).
__global__ void __launch_bounds__(kEntryThreads) k_rotate_emit(StepParams p) {
  pdl_wait();
  pdl_launch();
  if (block_skips(p.status)) return;
  const Geometry &geo = p.geo;
  if (blockIdx.x >= p.emit_blocks) {
    if (geo.exact) return;  // no ring under exact LRU
    const Bitmap bucket = class_bitmap(p.grp, geo, p.cur);
    const Bitmap cold = class_bitmap(p.grp, geo, geo.B);
    const uint32_t nthr = (gridDim.x - p.emit_blocks) * blockDim.x;
    const uint32_t t = (blockIdx.x - p.emit_blocks) * blockDim.x + threadIdx.x;
    for (uint32_t w = t; w < geo.gd.n0; w += nthr) {
      const uint32_t b = bucket.w0[w];
      if (b) {
        const uint32_t c = cold.w0[w];
        cold.w0[w] = c | b;
        bucket.w0[w] = 0;
        if (c == 0) {
          const uint32_t old1 = atomicOr(&cold.w1[w >> 5], 1u << (w & 31));
          if (old1 == 0) atomicOr(&cold.w2[w >> 10], 1u << ((w >> 5) & 31));
        }
      }
    }
    for (uint32_t w = t; w < geo.gd.n1; w += nthr) {
      const uint32_t moved = bucket.cnt[w];  // disjoint classes: counts add
      if (moved) {
        cold.cnt[w] += moved;
        bucket.cnt[w] = 0;
      }
      bucket.w1[w] = 0;
    }
    for (uint32_t w = t; w < geo.gd.n2; w += nthr) bucket.w2[w] = 0;
    return;
  }
  const uint32_t e = blockIdx.x * blockDim.x + threadIdx.x;
  const Flags f = entry_flags(p, e);
  __shared__ uint32_t sf[kEntryThreads / 32], sm[kEntryThreads / 32];
  const uint32_t incf = warp_incl_scan(f.first), incm = warp_incl_scan(f.miss);
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  if (lane == 31) {
    sf[warp] = incf;
    sm[warp] = incm;
  }
  __syncthreads();
  uint32_t bf = p.blk[blockIdx.x].x, bmiss = p.blk[blockIdx.x].y;
  for (uint32_t w = 0; w < warp; ++w) {
    bf += sf[w];
    bmiss += sm[w];
  }
  const uint32_t pos = bf + incf - f.first;    // exclusive: unique rows before e
  const uint32_t mpos = bmiss + incm - f.miss; // exclusive: misses before e
  if (e < p.E && (e % p.QK) == 0) p.req_off[e / p.QK] = (int32_t)pos;
  if (!f.first) return;
  p.grp.uniq[pos] = f.a;
  p.addr_row[f.a] = pos;
  if (f.miss) {
    p.miss_list[mpos] = f.a;
    if (p.geo.cache) {  // the owner partition's GPU slot (resident after the owner's step)
      const uint32_t part = f.a % p.src.P;
      const uint32_t om = part < kMaxParts ? p.src.map[part][f.a / p.src.P] : kNone;
      if ((om & kHostBit) || om >= (1u << kSrcShift)) latch(p.status, ULA_ERR_INTERNAL);
      p.miss_hs[mpos] = (part << kSrcShift) | (om & ((1u << kSrcShift) - 1u));
    } else {
      p.miss_hs[mpos] = f.m & kSlotMask;
    }
    p.miss_row[mpos] = pos;
    p.grp.row_slot[pos] = kNone;  // filled (and its output written) by the move
  } else if (f.m >= geo.S) {
    latch(p.status, ULA_ERR_INTERNAL);
  } else {
    // (3b) a hit: its slot for the gather, its access in this round, and (PB-LRU)
    // its bit in the step's hit map, which the marking applies to the labels
    p.grp.row_slot[pos] = f.m;
    p.grp.stamp[f.m] = p.round;
    if (!geo.exact) atomicOr(&p.grp.hitbits[f.m >> 5], 1u << (f.m & 31));
  }
}

// (4) Walk the segment counts of the classes in `ord` for the first `quota` set
// bits, then the host-free bitmap for the first K = quota - (free slots taken)
// set bits, and record one work entry per segment that holds some of them.
// Block-wide (T threads); stops as soon as the quota is met.
// One step of the walk over segment counts cnt[s0 .. s0 + T*V): threads take V
// consecutive segments each; segments holding ranks below `rem` (counted from
// `base`) become work entries (position y).  Advances base/rem; returns what it took.
template <int T>
__device__ __forceinline__ uint32_t walk_chunk(const uint32_t *cnt, uint32_t nseg, uint32_t s0,
                                               uint32_t y, uint32_t &base, uint32_t &rem,
                                               uint4 *work, uint32_t *s_nwork) {
  uint32_t v[kWalkSegs];
  uint32_t mine = 0;
  const uint32_t first = s0 + threadIdx.x * kWalkSegs;
#pragma unroll
  for (int j = 0; j < kWalkSegs; ++j) {
    v[j] = first + j < nseg ? __ldcg(&cnt[first + j]) : 0u;
    mine += v[j];
  }
  uint32_t total, ntake;
  uint32_t excl = block_incl_scan<T>(mine, &total) - mine;
  uint32_t takes = 0;
  {  // this thread's segments that hold ranks below rem
    uint32_t e = excl;
#pragma unroll
    for (int j = 0; j < kWalkSegs; ++j) {
      takes += (v[j] > 0 && e < rem) ? 1u : 0u;
      e += v[j];
    }
  }
  uint32_t pos = block_incl_scan<T>(takes, &ntake) - takes + *s_nwork;
#pragma unroll
  for (int j = 0; j < kWalkSegs; ++j) {
    if (v[j] > 0 && excl < rem) work[pos++] = make_uint4(y, first + j, base + excl, v[j]);
    excl += v[j];
  }
  const uint32_t got = min(total, rem);
  base += got;
  rem -= got;
  __syncthreads();
  if (threadIdx.x == 0) *s_nwork += ntake;
  __syncthreads();
  return got;
}

// (4) Walk the segment counts of the classes in `ord` for the first `quota` set
// bits, then the host-free bitmap for the first K = total - (free slots taken)
// set bits (a step's victims that hold data; alloc: what the GPU walk lacked),
// and record one work entry per segment that holds some of them.  Block-wide (T
// threads); stops as soon as the quota is met.  A step walks for quota = total
// victims under PB-LRU; under exact LRU it walks the free class only, for
// quota = min(total, free slots), and the scan picks the rest.
template <int T>
__device__ void select_walk(const GroupDev &g, const Geometry &geo, const Order &ord,
                            uint32_t quota, uint32_t total, bool is_step, int *status) {
  __shared__ uint32_t s_nwork;
  if (threadIdx.x == 0) s_nwork = 0;
  __syncthreads();
  uint32_t rem = quota, base = 0, taken_free = 0, taken_cold = 0;
  const uint32_t free_gpu = __ldcg(&g.cnt->free_gpu);
  for (uint32_t y = 0; y < ord.n_cls && rem > 0; ++y) {
    if (ord.cls[y] == geo.B + 1 && free_gpu == 0) continue;  // no free slot to walk
    const Bitmap bm = class_bitmap(g, geo, ord.cls[y]);
    uint32_t taken_y = 0;
    for (uint32_t s0 = 0; s0 < geo.nseg && rem > 0; s0 += T * kWalkSegs)
      taken_y += walk_chunk<T>(bm.cnt, geo.nseg, s0, y, base, rem, g.work, &s_nwork);
    if (ord.cls[y] == geo.B + 1) taken_free += taken_y;
    else if (ord.cls[y] == geo.B) taken_cold += taken_y;
  }
  const uint32_t F = taken_free;
  const uint32_t nwork_gpu = s_nwork;
  // (a local buffer writes nothing back: its victims' copies are dropped)
  const uint32_t K = geo.cache ? 0u : (is_step && rem == 0) ? total - F : (is_step ? 0u : rem);
  uint32_t hrem = K, hbase = 0;
  const Bitmap hb = host_free_bitmap(g);
  for (uint32_t s0 = 0; s0 < geo.hseg && hrem > 0; s0 += T * kWalkSegs)
    walk_chunk<T>(hb.cnt, geo.hseg, s0, kHostPos, hbase, hrem, g.work, &s_nwork);
  if (threadIdx.x != 0) return;
  GroupCounters *c = g.cnt;
  if ((is_step && rem > 0) || hrem > 0) {
    latch(status, ULA_ERR_INTERNAL);  // the capacity check rules this out
    return;
  }
  c->F = F;
  c->K = K;
  c->n_work = s_nwork;
  c->n_work_gpu = nwork_gpu;
  if (is_step) {
    c->free_gpu -= F;   // F free slots filled
    if (!geo.cache) c->free_host += F;  // K host slots taken, quota host slots released
    c->stat[kStVictFree] += F;
    if (geo.exact) {
      c->stat[kStVictCold] += total - F;  // occupied slots (the scan's victims)
    } else {
      c->stat[kStVictCold] += taken_cold;
      c->stat[kStVictRing] += quota - F - taken_cold;
    }
    c->stat[kStWriteback] += K;
    c->stat[kStBytesD2H] += (unsigned long long)K * g.layers * geo.W;
  } else {
    c->free_gpu -= F;
    c->free_host -= K;
  }
}

// (3b) Every hit moves to the current bucket (labels only), applied word by word:
// one warp per segment takes the step's hit map for its 32 words and, class by
// class, clears the hit bits on every other class and sets them on the current
// bucket, then rewrites the segment's count and level-1 word (the warp owns both
// for every class) and flips the level-2 bit if the segment's emptiness changed.
// The hit map is cleared on the way.  (Exact LRU: hits only restamp, done by the
// compaction.)  The last block then walks the classes for the M victims (exact
// LRU: the free class only).
__global__ void __launch_bounds__(kEntryThreads) k_mark_select(StepParams p) {
  pdl_wait();
  pdl_launch();
  if (block_skips(p.status)) return;
  const GroupDev &g = p.grp;
  const Geometry &geo = p.geo;
  if (!geo.exact) {
    const uint32_t lane = lane_id();
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    for (uint32_t sg = warp; sg < geo.nseg; sg += nwarps) {
      const uint32_t w = sg * 32 + lane;
      const bool valid = w < geo.gd.n0;
      const uint32_t hw = valid ? g.hitbits[w] : 0u;
      if (!__any_sync(0xffffffffu, hw != 0)) continue;
      if (hw) g.hitbits[w] = 0;
      for (uint32_t c0 = 0; c0 < geo.B + 2; c0 += kMarkClasses) {
        uint32_t xs[kMarkClasses];
#pragma unroll
        for (int u = 0; u < kMarkClasses; ++u) {  // the classes' words, loaded at once
          const uint32_t c = c0 + u;
          xs[u] = valid && c < geo.B + 2 ? class_bitmap(g, geo, c).w0[w] : 0u;
        }
#pragma unroll
        for (int u = 0; u < kMarkClasses; ++u) {
          const uint32_t c = c0 + u;
          if (c >= geo.B + 2) break;
          const Bitmap bm = class_bitmap(g, geo, c);
          const uint32_t x = xs[u];
          if (c == geo.B + 1) {  // a hit's slot is never free
            if (x & hw) latch(p.status, ULA_ERR_INTERNAL);
            continue;
          }
          const uint32_t nx = c == p.cur ? (x | hw) : (x & ~hw);
          if (!__any_sync(0xffffffffu, nx != x)) continue;
          if (nx != x) bm.w0[w] = nx;
          int d = (int)__popc(nx) - (int)__popc(x);
#pragma unroll
          for (int o = 16; o; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
          const uint32_t nz = __ballot_sync(0xffffffffu, nx != 0);
          if (lane == 0) {
            bm.cnt[sg] += (uint32_t)d;
            const uint32_t old1 = bm.w1[sg];
            if (nz != old1) {
              bm.w1[sg] = nz;
              const uint32_t bit = 1u << (sg & 31);
              if (old1 == 0) atomicOr(&bm.w2[sg >> 5], bit);       // segment became non-empty
              else if (nz == 0) atomicAnd(&bm.w2[sg >> 5], ~bit);  // segment became empty
            }
          }
        }
      }
    }
  }
  if (!last_block(&g.cnt->done[1])) return;
  const uint32_t M = __ldcg(&g.cnt->M);
  const uint32_t quota = geo.exact ? min(M, __ldcg(&g.cnt->free_gpu)) : M;
  select_walk<kEntryThreads>(g, geo, p.order, quota, M, true, p.status);
}

// (5) The order in which the move runs the fills: miss indices [0, M) sorted by
// bucket of their host slot (host slot >> fill_shift, kFillBuckets buckets; any order
// inside a bucket), one block.  The pairing of miss i with victim i is unchanged;
// only the order of the copies changes, so that at any moment the move's warps read
// a narrow, advancing window of the host pool instead of all of it at random (the
// GPU keeps too few address translations for random 2.6 KB reads over tens of GB of
// host memory).  The write-backs need no sort: the j-th victim that holds data goes to
// the j-th lowest free host slot, so victim order is host-address order already.
constexpr int kOrderThreads = 256;

// One range [lo, hi) of miss indices, sorted into fill_order[lo, hi).
__device__ void fill_order_range(const EmitParams &p, uint32_t lo, uint32_t hi, uint32_t *hist) {
  const uint32_t shift = p.geo.fill_shift;
  const uint32_t lane = lane_id();
  for (uint32_t b = threadIdx.x; b < kFillBuckets; b += kOrderThreads) hist[b] = 0;
  __syncthreads();
  // lanes of a warp with the same bucket (neighbouring misses often share one) take
  // their positions with one atomic
  auto claim = [&](uint32_t i0) -> uint32_t {  // position of miss i0 + threadIdx.x, or kNone
    const uint32_t i = i0 + threadIdx.x;
    const bool act = i < hi;
    const uint32_t b = act ? min(__ldcg(&p.miss_hs[i]) >> shift, kFillBuckets - 1) : kNone;
    const uint32_t peers = __match_any_sync(0xffffffffu, b);
    const uint32_t leader = __ffs(peers) - 1;
    uint32_t base = 0;
    if (act && lane == leader) base = atomicAdd(&hist[b], (uint32_t)__popc(peers));
    base = __shfl_sync(0xffffffffu, base, leader);
    return act ? base + __popc(peers & ((1u << lane) - 1u)) : kNone;
  };
  for (uint32_t i0 = lo; i0 < hi; i0 += kOrderThreads) claim(i0);  // bucket sizes
  __syncthreads();
  constexpr uint32_t kPer = kFillBuckets / kOrderThreads;
  uint32_t v[kPer], mine = 0;
#pragma unroll
  for (uint32_t j = 0; j < kPer; ++j) {
    v[j] = hist[threadIdx.x * kPer + j];
    mine += v[j];
  }
  uint32_t total;
  uint32_t run = lo + block_incl_scan<kOrderThreads>(mine, &total) - mine;
#pragma unroll
  for (uint32_t j = 0; j < kPer; ++j) {
    hist[threadIdx.x * kPer + j] = run;  // exclusive start of each bucket
    run += v[j];
  }
  __syncthreads();
  for (uint32_t i0 = lo; i0 < hi; i0 += kOrderThreads) {
    const uint32_t pos = claim(i0);
    if (pos != kNone) p.fill_order[pos] = i0 + threadIdx.x;
  }
  __syncthreads();
}

// The misses made resident [0, M), then those the overflow bypass reads in place
// [M, M + Mx), each range in host-slot bucket order.
__device__ void fill_order_block(const EmitParams &p, const GroupDev &g) {
  __shared__ uint32_t hist[kFillBuckets];
  const uint32_t M = __ldcg(&g.cnt->M), Mx = __ldcg(&g.cnt->Mx);
  fill_order_range(p, 0, M, hist);
  if (Mx) fill_order_range(p, M, M + Mx, hist);
}

// (4) Each work entry's segment: its set bits in ascending order get the ranks
// [base, base + count); ranks below the quota are written out.  Host entries
// claim their slots (clears only on the host-free bitmap; GPU classes read only).
// With a fill order to compute (a step), the grid has one more block, which does that.
__global__ void __launch_bounds__(kOrderThreads) k_select_emit(EmitParams p) {
  pdl_wait();
  pdl_launch();
  if (*(volatile int *)p.status) return;
  const GroupDev g = p.groups[p.group0 + blockIdx.y];
  const uint32_t nblk = p.fill_order ? gridDim.x - 1 : gridDim.x;  // blocks that emit
  if (blockIdx.x >= nblk) {
    fill_order_block(p, g);
    span_close(p.span);
    return;
  }
  const Geometry &geo = p.geo;
  const GroupCounters *c = g.cnt;
  const uint32_t n_work = c->n_work;
  const uint32_t q_gpu = p.quota == 0xffffffffu ? (geo.exact ? c->F : c->M) : p.quota;
  const uint32_t q_host = c->K;
  const uint32_t lane = lane_id();
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t nwarps = (nblk * blockDim.x) >> 5;
  for (uint32_t i = warp; i < n_work; i += nwarps) {
    const uint4 e = g.work[i];
    const bool host = e.x == kHostPos;
    if (!host && e.x >= p.order.n_cls) {
      if (lane == 0) latch(p.status, ULA_ERR_INTERNAL);
      continue;
    }
    const Bitmap bm = host ? host_free_bitmap(g) : class_bitmap(g, geo, p.order.cls[e.x]);
    const uint32_t n0 = host ? geo.hd.n0 : geo.gd.n0;
    const uint32_t q = host ? q_host : q_gpu;
    uint32_t *dst = host ? g.wb_host : g.victims;
    const uint32_t seg = e.y;
    const uint32_t wi = seg * 32 + lane;
    const uint32_t s1 = bm.w1[seg];  // level-1 summary: which words of the segment hold bits
    uint32_t word = (((s1 >> lane) & 1u) && wi < n0) ? bm.w0[wi] : 0u;
    const uint32_t pc = __popc(word);
    uint32_t rank = e.z + warp_incl_scan(pc) - pc;
    uint32_t taken = 0;
    while (word && rank < q) {
      const uint32_t b = __ffs(word) - 1;
      word &= word - 1;
      taken |= 1u << b;
      dst[rank++] = wi * 32 + b;
    }
    if (host && taken) bm_clear_mask(bm, wi, taken);  // claim the write-back targets
  }
  span_close(p.span);
}

// -------------------------------------------------------- move and commit
//
// (5) Data first: per victim i (one warp), write the victim's rows back to its
// host slot if it holds data and fill miss i's rows from its host slot; for the
// missed row, its outputs are written straight from the moved bytes (6).  Each
// lane handles the same 16-byte chunks in the write-back and in the fill, so
// its read of a chunk precedes its write of the same chunk.  Host memory is
// reached directly over the host link.  The per-victim plan (victim slot, host
// slots, row) is read up front from arrays filled by the compaction and the
// selection, so a warp starts its copies after one round of independent loads.
// Once a warp's copies of victim i are done, its lane 0 commits victim i's map
// and labels (the readers of the map are later kernels).
// (5) The map after the data: victim i's old owner now maps to its host slot (a
// local buffer drops it), miss i to the victim slot; the slot joins the current
// bucket (clears on its old class, sets on cur); the miss's host slot is released
// (sets only on the host-free bitmap).  Called once victim i's copies are done.
__device__ __forceinline__ void commit_victim(const MoveParams &p, uint32_t i, uint32_t F) {
  const GroupDev &g = p.grp;
  const Geometry &geo = p.geo;
  const uint32_t v = g.victims[i];
  const uint32_t a = p.miss_list[i];
  const uint32_t hs = p.miss_hs[i];
  const bool owned = !geo.cache && i >= F;
  const uint32_t hd = owned ? g.wb_host[i - F] : 0u;
  const uint32_t o = v < geo.S ? g.owner[v] : kNone;
  const bool bad = geo.cache ? (o != kNone && o >= geo.max_logical)
                             : (hs >= geo.H || (owned ? (hd >= geo.H || o >= geo.max_logical)
                                                      : o != kNone));
  if (v >= geo.S || a >= geo.max_logical || bad) {
    latch(p.status, ULA_ERR_INTERNAL);
    return;
  }
  if (owned) g.map[o] = kHostBit | hd;
  else if (geo.cache && o != kNone) g.map[o] = kUnalloc;  // the buffer's old copy is dropped
  g.map[a] = v;
  g.owner[v] = a;
  const uint32_t c = slot_class(geo, g.stamp[v], p.round);
  const uint32_t to = access_class(geo, p.cur);
  if (c != to) {
    bm_clear(class_bitmap(g, geo, c), v);
    bm_set(class_bitmap(g, geo, to), v);
  }
  g.stamp[v] = p.round;
  if (!geo.cache) bm_set(host_free_bitmap(g), hs);
}

// (1) every entry's unique row (grid-stride over the selection)
__device__ __forceinline__ void write_entry_rows(const MoveParams &p) {
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < p.E; e += stride) {
    const uint32_t a = p.sel[e];
    p.entry_row[e] = a == kPad ? -1 : (int32_t)p.addr_row[a];
  }
}

constexpr int kMoveUnroll = ULA_MOVE_UNROLL;
constexpr int kMoveThreads = ULA_MOVE_THREADS;

// (5) Before the move: the rows of every victim that holds data (victims F..M-1) are
// copied to the staging area, one warp per victim (HBM to HBM).  The move then writes
// victims back from the staging area and fills them, each in its own order, with no
// ordering between a victim's write-back and its fill.
__global__ void __launch_bounds__(256) k_stage(MoveParams p) {
  pdl_launch();  // the move may be scheduled early (it waits for this kernel to finish)
  if (*(volatile int *)p.status) return;
  const GroupDev &g = p.grp;
  const Geometry &geo = p.geo;
  span_open(p.span);
  write_entry_rows(p);  // (1) every entry's unique row
  if (geo.cache || !p.stage) {  // a local buffer writes nothing back
    span_close(p.span);
    return;
  }
  const uint32_t M = g.cnt->M, F = g.cnt->F;
  const uint32_t lane = lane_id();
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
  const size_t sb = (size_t)g.layers * geo.W;
  const uint32_t nvec = (uint32_t)(sb / 16);
  for (uint32_t i = F + warp; i < M; i += nwarps) {
    const uint32_t v = g.victims[i];
    if (v >= geo.S) {
      if (lane == 0) latch(p.status, ULA_ERR_INTERNAL);
      continue;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(g.gpu_pool + (size_t)v * sb);
    uint4 *dst = reinterpret_cast<uint4 *>(p.stage + (size_t)(i - F) * sb);
    for (uint32_t c0 = 0; c0 < nvec; c0 += 32 * kMoveUnroll) {
      uint4 x[kMoveUnroll];
#pragma unroll
      for (int u = 0; u < kMoveUnroll; ++u) {
        const uint32_t c = c0 + u * 32 + lane;
        if (c < nvec) x[u] = __ldcs(src + c);
      }
#pragma unroll
      for (int u = 0; u < kMoveUnroll; ++u) {
        const uint32_t c = c0 + u * 32 + lane;
        if (c < nvec) dst[c] = x[u];
      }
    }
  }
  span_close(p.span);
}

// One of victim x's copies is done (its write-back, or the fill of its miss); the
// last one commits x (a victim that holds data has two, a free slot or a local
// buffer's victim one).  Called by one lane per completed copy, after a fence that
// orders the warp's copy writes before it.
__device__ __forceinline__ void copy_done(const MoveParams &p, uint32_t x, uint32_t F) {
  const bool two = !p.geo.cache && x >= F;
  if (two) {
    if (atomicAdd(&p.vdone[x], 1u) != 1u) return;  // the other copy is still running
    p.vdone[x] = 0;                                   // ready for the next step
  }
  commit_victim(p, x, F);
}

// (5) Data first: task t (one warp) writes victim t's staged rows back to its host
// slot if it holds data (victim order = ascending host slots), and fills miss
// i = fill_order[t] (host-slot bucket order) from its host slot into victim i's GPU
// slot, writing the missed row's outputs (6) from the moved bytes.  Both directions of
// the host link are busy in every warp.  Host memory is reached directly over the host
// link.  Completed copies are counted per victim; the lanes of a warp commit up to 32
// victims at a time, each once both of its copies are done (the map after the data).
constexpr uint32_t kCommitBatch = 16;  // tasks per warp between commit rounds (2 copies each)

__global__ void __launch_bounds__(kMoveThreads, ULA_MOVE_MINBLOCKS) k_move(MoveParams p) {
  pdl_wait();  // (no early trigger: the commit's blocks would hold SM room for the whole move)
  if (*(volatile int *)p.status) return;
  span_open(p.span);
  const GroupDev &g = p.grp;
  const Geometry &geo = p.geo;
  const uint32_t M = g.cnt->M, F = g.cnt->F, Mx = g.cnt->Mx;
  const uint32_t lane = lane_id();
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
  const size_t sb = (size_t)g.layers * geo.W;
  const uint32_t nvec = (uint32_t)(sb / 16);
  const uint32_t CW = geo.W / 16;
  uint4 *out = reinterpret_cast<uint4 *>(p.out);
  // overflow bypass: misses [M, M + Mx) are copied from their host slots to the
  // output only (they stay on the host), in host-slot bucket order as well
  for (uint32_t t = M + warp; t < M + Mx; t += nwarps) {
    const uint32_t i = p.fill_order[t];
    const bool bad_i = i < M || i >= M + Mx;
    const uint32_t hs = bad_i ? kNone : p.miss_hs[i];
    const uint32_t row = bad_i ? kNone : p.miss_row[i];
    if (bad_i || !out || hs >= geo.H || row >= p.out_cap) {
      if (lane == 0) latch(p.status, ULA_ERR_INTERNAL);
      continue;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(g.host_pool + (size_t)hs * sb);
    for (uint32_t c0 = 0; c0 < nvec; c0 += 32 * kMoveUnroll) {
      uint4 v[kMoveUnroll];
#pragma unroll
      for (int u = 0; u < kMoveUnroll; ++u) {
        const uint32_t c = c0 + u * 32 + lane;
        if (c < nvec) v[u] = src[c];
      }
#pragma unroll
      for (int u = 0; u < kMoveUnroll; ++u) {
        const uint32_t c = c0 + u * 32 + lane;
        if (c < nvec) {
          const uint32_t j = c / CW;
          out[((size_t)j * p.out_cap + row) * CW + (c - j * CW)] = v[u];
        }
      }
    }
  }
  uint32_t mine = kNone;  // the victim whose copy this lane reports at the next commit round
  uint32_t batch = 0;
  auto commit_round = [&]() {
    __threadfence();  // this lane's copy writes before any commit that counts them
    __syncwarp();
    if (mine != kNone) copy_done(p, mine, F);
    mine = kNone;
    batch = 0;
    __syncwarp();
  };
  for (uint32_t t = warp; t < M; t += nwarps) {
    const bool back = !geo.cache && t >= F;  // (a local buffer drops its victims' copies)
    const uint32_t hd = back ? g.wb_host[t - F] : 0u;
    const uint32_t i = p.fill_order[t];
    const bool bad_i = i >= M;
    const uint32_t v = bad_i ? kNone : g.victims[i];
    const uint32_t hs = bad_i ? kNone : p.miss_hs[i];
    const uint32_t row = bad_i ? kNone : p.miss_row[i];
    // the fill's source: the miss's host slot, or (local buffer) its owner partition's GPU slot
    const uint32_t part = hs >> kSrcShift, pslot = hs & ((1u << kSrcShift) - 1u);
    const bool src_bad = geo.cache ? (part >= p.src.P || pslot >= p.src.S) : hs >= geo.H;
    if (bad_i || v >= geo.S || src_bad || (back && (hd >= geo.H || !p.stage)) ||
        (out && row >= p.out_cap)) {
      if (lane == 0) latch(p.status, ULA_ERR_INTERNAL);
      continue;
    }
    uint4 *gp = reinterpret_cast<uint4 *>(g.gpu_pool + (size_t)v * sb);
    const uint4 *src = reinterpret_cast<const uint4 *>(
        geo.cache ? p.src.pool[part] + (size_t)pslot * sb : g.host_pool + (size_t)hs * sb);
    const uint4 *bsrc =
        back ? reinterpret_cast<const uint4 *>(p.stage + (size_t)(t - F) * sb) : nullptr;
    uint4 *bdst = back ? reinterpret_cast<uint4 *>(g.host_pool + (size_t)hd * sb) : nullptr;
    for (uint32_t c0 = 0; c0 < nvec; c0 += 32 * kMoveUnroll) {
      uint4 fill[kMoveUnroll], wb[kMoveUnroll];
#pragma unroll
      for (int u = 0; u < kMoveUnroll; ++u) {
        const uint32_t c = c0 + u * 32 + lane;
        if (c < nvec) fill[u] = src[c];
      }
      if (back) {
#pragma unroll
        for (int u = 0; u < kMoveUnroll; ++u) {
          const uint32_t c = c0 + u * 32 + lane;
          if (c < nvec) wb[u] = __ldcs(bsrc + c);
        }
#pragma unroll
        for (int u = 0; u < kMoveUnroll; ++u) {
          const uint32_t c = c0 + u * 32 + lane;
          if (c < nvec) bdst[c] = wb[u];
        }
      }
#pragma unroll
      for (int u = 0; u < kMoveUnroll; ++u) {
        const uint32_t c = c0 + u * 32 + lane;
        if (c < nvec) gp[c] = fill[u];
      }
      if (out) {  // (6) the missed row's outputs, from the moved bytes
#pragma unroll
        for (int u = 0; u < kMoveUnroll; ++u) {
          const uint32_t c = c0 + u * 32 + lane;
          if (c < nvec) {
            const uint32_t j = c / CW;
            out[((size_t)j * p.out_cap + row) * CW + (c - j * CW)] = fill[u];
          }
        }
      }
    }
    // report both copies of this task at the next commit round (lanes 2b, 2b + 1)
    if (lane == 2 * batch) mine = back ? t : kNone;
    if (lane == 2 * batch + 1) mine = i;
    if (++batch == kCommitBatch) commit_round();
  }
  commit_round();
  span_close(p.span);
}

// (5) With the per-layer signal: the same moves, layer by layer.  The chunks of
// every layer (16 bytes each, CW per row; layer 0 of every miss and every bypassed
// miss first, then layer 1, ...) are handed out in order, kMoveBatch at a time, from
// a counter, so the chunks of layer j are all taken before any of layer j + 1 and
// layer j completes soon after its last batch was taken.  Inside a batch
// consecutive lanes take consecutive chunks; a lane reads the victim's chunk
// (write-back) and the miss's chunk (fill) before it writes either, so each chunk
// leaves before the new one lands.  Completed chunks are counted per layer; the
// warp that completes layer j gives the move's contribution to the layer's signal.
constexpr int kMoveLayerUnroll = 4;
#ifndef ULA_MOVE_BATCH
#define ULA_MOVE_BATCH (32 * 4 * 2)
#endif
constexpr uint32_t kMoveBatch = ULA_MOVE_BATCH;  // chunks handed out at a time (a multiple of 32)

__global__ void __launch_bounds__(256, 3) k_move_layers(MoveParams p) {
  pdl_wait();
  if (*(volatile int *)p.status) return;
  const GroupDev &g = p.grp;
  const Geometry &geo = p.geo;
  const uint32_t M = g.cnt->M, F = g.cnt->F, Mx = g.cnt->Mx;
  const uint32_t L = g.layers;
  const uint32_t CW = geo.W / 16;
  const size_t sb = (size_t)L * geo.W;
  const uint32_t lane = lane_id();
  const uint32_t per_layer = (M + Mx) * CW;  // chunks of one layer
  const uint32_t total = per_layer * L;
  const uint32_t needed = p.out ? 2u : 1u;
  uint4 *out = reinterpret_cast<uint4 *>(p.out);
  if (per_layer == 0) {  // nothing to move: the move's contribution to every layer
    if (blockIdx.x == 0 && threadIdx.x == 0)
      for (uint32_t j = 0; j < L; ++j) layer_contrib(g, j, needed, p.round);
    return;
  }
  uint32_t *next = &g.move_done[L];  // the dispenser (reset before the step's move)
  for (;;) {
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(next, kMoveBatch);
    base = __shfl_sync(0xffffffffu, base, 0);
    if (base >= total) break;
    const uint32_t end = min(base + kMoveBatch, total);
    for (uint32_t c0 = base + lane; c0 < end; c0 += 32 * kMoveLayerUnroll) {
      uint4 fill[kMoveLayerUnroll], back[kMoveLayerUnroll];
      uint32_t vs[kMoveLayerUnroll], hds[kMoveLayerUnroll], rows[kMoveLayerUnroll],
          offs[kMoveLayerUnroll], js[kMoveLayerUnroll];
#pragma unroll
      for (int u = 0; u < kMoveLayerUnroll; ++u) {
        vs[u] = hds[u] = rows[u] = kNone;
        offs[u] = js[u] = 0;
        const uint32_t c = c0 + u * 32;
        if (c >= end) continue;
        const uint32_t j = c / per_layer, cc = c - j * per_layer;
        const uint32_t i = cc / CW, k = cc - i * CW;
        const uint32_t hs = p.miss_hs[i], row = p.miss_row[i];
        if (hs >= geo.H || (out && row >= p.out_cap) || (i >= M && !out)) {
          latch(p.status, ULA_ERR_INTERNAL);
          continue;
        }
        uint32_t v = kNone, hd = kNone;
        if (i < M) {  // resident miss: the victim slot, and its write-back target if it holds data
          v = g.victims[i];
          if (i >= F) hd = g.wb_host[i - F];
          if (v >= geo.S || (i >= F && hd >= geo.H)) {
            latch(p.status, ULA_ERR_INTERNAL);
            continue;
          }
        }
        const uint32_t off = j * geo.W + 16 * k;  // byte offset inside a slot
        js[u] = j;
        offs[u] = off;
        vs[u] = v;
        hds[u] = hd;
        rows[u] = out ? row : kNone;
        fill[u] = *reinterpret_cast<const uint4 *>(g.host_pool + (size_t)hs * sb + off);
        if (hd != kNone) back[u] = *reinterpret_cast<const uint4 *>(g.gpu_pool + (size_t)v * sb + off);
      }
#pragma unroll
      for (int u = 0; u < kMoveLayerUnroll; ++u) {
        if (hds[u] != kNone)
          *reinterpret_cast<uint4 *>(g.host_pool + (size_t)hds[u] * sb + offs[u]) = back[u];
        if (vs[u] != kNone)
          *reinterpret_cast<uint4 *>(g.gpu_pool + (size_t)vs[u] * sb + offs[u]) = fill[u];
        if (rows[u] != kNone)
          out[((size_t)js[u] * p.out_cap + rows[u]) * CW + (offs[u] - js[u] * geo.W) / 16] = fill[u];
      }
    }
    __threadfence();  // every lane's writes of the batch before its count
    __syncwarp();
    if (lane == 0) {
      for (uint32_t j = base / per_layer; j <= (end - 1) / per_layer; ++j) {
        const uint32_t n = min(end, (j + 1) * per_layer) - max(base, j * per_layer);
        if (atomicAdd(&g.move_done[j], n) + n == per_layer) {
          g.move_done[j] = 0;
          layer_contrib(g, j, needed, p.round);
        }
      }
    }
  }
}

// (5) Then the map: one thread per victim, after every copy has completed
// (kernel boundary).  The evicted owner now maps to its host slot, the miss to
// the victim slot; the slot joins the current bucket (clears on its old class,
// sets on cur); the miss's host slot is released (sets only on the host-free
// bitmap).  (1) The idle threads also write every entry's unique row.
__global__ void k_commit(MoveParams p) {
  pdl_wait();
  if (*(volatile int *)p.status) return;
  const uint32_t M = p.grp.cnt->M, F = p.grp.cnt->F;
  const uint32_t stride = gridDim.x * blockDim.x;
  write_entry_rows(p);
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < M; i += stride)
    commit_victim(p, i, F);
}

// ------------------------------------------------------------------ gather
//
// (6) out[j][u] = layer j of unique row u's slot for the layers j of this launch,
// [layer, layer + nlayers), for the rows that hit (recorded by the marking; a hit's
// slot does not change in its round, so this may run while the misses are being moved;
// missed rows are written by the move).  A slot holds its layers' rows back to back,
// so the launch reads nlayers * W contiguous bytes per slot.  Two kernels: the bulk
// gather below (rows that fit its per-thread buffers), and this one, with registers,
// for longer rows.  The U rows are spread
// over all warps (rows_per_warp = ceil(U / warps), at most 32): lanes read the warp's
// slots, then the warp streams the rows' 16-byte chunks, consecutive lanes on
// consecutive chunks (coalesced within a slot; per layer, the warp's output rows are
// contiguous).  Loads are issued kGatherUnroll deep before the stores.
constexpr int kGatherUnroll = ULA_GATHER_UNROLL;

__global__ void __launch_bounds__(kGatherThreads, ULA_GATHER_MINBLOCKS) k_gather(GatherParams p) {
  if (*(volatile int *)p.status) return;
  span_open(p.span);
  const GroupDev &g = p.grp;
  const Geometry &geo = p.geo;
  const uint32_t U = g.cnt->U;
  if (U > p.out_cap) {  // only a re-gather into a short buffer can get here
    if (blockIdx.x == 0 && threadIdx.x == 0) latch(p.status, ULA_ERR_CAPACITY);
    return;
  }
  const uint32_t lane = lane_id();
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
  const uint32_t CW = geo.W / 16;
  const uint32_t NL = p.nlayers;
  const uint32_t RW = NL * CW;                 // chunks per slot in this launch
  const size_t sbv = (size_t)g.layers * CW;  // slot stride in uint4
  const size_t lsv = (size_t)p.out_cap * CW;  // output layer stride in uint4
  const uint4 *pool = reinterpret_cast<const uint4 *>(g.gpu_pool) + (size_t)p.layer * CW;
  uint4 *out = reinterpret_cast<uint4 *>(p.out) + (size_t)p.layer * lsv;
  uint32_t rpw = (U + nwarps - 1) / nwarps;
  rpw = rpw < 1 ? 1 : (rpw > 32 ? 32 : rpw);
  // chunk f = lane of a warp's rows: row r0, layer j0, column c0
  const uint32_t r0 = lane / RW, j0 = (lane % RW) / CW, c0 = lane % CW;
  for (uint32_t row0 = warp * rpw; row0 < U; row0 += nwarps * rpw) {
    const uint32_t nrows = min(rpw, U - row0);
    uint32_t slot = kNone;
    bool bad = false;
    if (lane < nrows) {
      const uint32_t m = g.row_slot[row0 + lane];
      bad = m != kNone && m >= geo.S;
      slot = bad ? kNone : m;
    }
    if (__any_sync(0xffffffffu, bad)) {
      if (lane == 0) latch(p.status, ULA_ERR_INTERNAL);
      continue;
    }
    const uint32_t total = nrows * RW;
    uint4 *orow = out + (size_t)row0 * CW;
    uint32_t r = r0, j = j0, c = c0;
    for (uint32_t f0 = 0; f0 < total; f0 += 32 * kGatherUnroll) {
      uint4 v[kGatherUnroll];
      const uint32_t rs = r, js = j, cs = c;
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u) {
        const uint32_t s = __shfl_sync(0xffffffffu, slot, r & 31);
        if (f0 + u * 32 + lane < total && s != kNone)
          v[u] = __ldcs(pool + (size_t)s * sbv + j * CW + c);
        c += 32;
        while (c >= CW) {
          c -= CW;
          if (++j == NL) {
            j = 0;
            ++r;
          }
        }
      }
      r = rs;
      j = js;
      c = cs;
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u) {
        const uint32_t s = __shfl_sync(0xffffffffu, slot, r & 31);
        if (f0 + u * 32 + lane < total && s != kNone) orow[j * lsv + (size_t)r * CW + c] = v[u];
        c += 32;
        while (c >= CW) {
          c -= CW;
          if (++j == NL) {
            j = 0;
            ++r;
          }
        }
      }
    }
  }
  span_close(p.span);
  // per-layer signal: the hit rows of a layer are one of its two contributions
  if (p.signal) {
    __threadfence();  // every thread's output writes before the block's ticket
    if (last_block(&g.gather_done[p.layer]) && threadIdx.x == 0)
      for (uint32_t j = p.layer; j < p.layer + NL; ++j) layer_contrib(g, j, 2u, p.round);
  }
}

// (6) The same gather with bulk copies (cp.async.bulk through shared memory), for
// slots that fit a thread's buffer: each thread moves whole rows -- one bulk load brings
// a hit row's layers [layer, layer + nlayers) (nlayers * W contiguous bytes of its slot)
// into the thread's buffer, completing on the thread's mbarrier; one bulk store per
// layer then writes the row to that layer's output plane; the thread's next load waits
// until those stores have read the buffer.  No row's bytes pass through registers and
// the load/store units stay free, so many rows are in flight per SM (kBulkThreads per
// block, several blocks per SM).  Threads take rows tid, tid + threads, ... of the
// unique rows; rows that missed are skipped (the move writes them).  Waits are bounded
// (1 s, then ULA_ERR_TIMEOUT).
constexpr int kBulkThreads = 16;
constexpr uint32_t kBulkBars = 128;  // the mbarriers' bytes at the head of shared memory

__device__ __forceinline__ uint32_t smem_u32(const void *ptr) {
  return (uint32_t)__cvta_generic_to_shared(ptr);
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  for (;;) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    if (done) return true;
    if (global_ns() - t0 > 1000000000ull) return false;
  }
}

__global__ void __launch_bounds__(kBulkThreads) k_gather_bulk(GatherParams p) {
  extern __shared__ __align__(128) uint8_t bulk_smem[];
  if (*(volatile int *)p.status) return;
  span_open(p.span);
  const GroupDev &g = p.grp;
  const Geometry &geo = p.geo;
  const uint32_t U = g.cnt->U;
  if (U > p.out_cap) {  // only a re-gather into a short buffer can get here
    if (blockIdx.x == 0 && threadIdx.x == 0) latch(p.status, ULA_ERR_CAPACITY);
    return;
  }
  const uint32_t W = geo.W, NL = p.nlayers, rb = NL * W;  // bytes per row moved
  const uint32_t bar = smem_u32(bulk_smem) + threadIdx.x * 8;
  const uint32_t buf = smem_u32(bulk_smem) + kBulkBars + threadIdx.x * rb;
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  const size_t sb = (size_t)g.layers * W;
  const uint8_t *pool = g.gpu_pool + (size_t)p.layer * W;
  uint8_t *out = p.out + (size_t)p.layer * p.out_cap * W;
  const uint32_t nthr = gridDim.x * blockDim.x;
  uint32_t next = blockIdx.x * blockDim.x + threadIdx.x;  // the next row this thread looks at
  // the next hit row at or after `next` (and its slot); false when none is left
  auto next_hit = [&](uint32_t &row, uint32_t &slot) -> bool {
    while (next < U) {
      const uint32_t r = next, m = g.row_slot[r];
      next += nthr;
      if (m == kNone) continue;  // a miss: written by the move
      if (m >= geo.S) {
        latch(p.status, ULA_ERR_INTERNAL);
        continue;
      }
      row = r;
      slot = m;
      return true;
    }
    return false;
  };
  auto load = [&](uint32_t slot) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(rb)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(buf), "l"(pool + (size_t)slot * sb), "r"(rb), "r"(bar)
        : "memory");
  };
  uint32_t row, slot, parity = 0;
  bool have = next_hit(row, slot);
  if (have) load(slot);
  while (have) {
    if (!mbar_wait(bar, parity)) {
      latch(p.status, ULA_ERR_TIMEOUT);
      mbar_wait(bar, parity);  // (once more, bounded, for the load still in flight)
      break;
    }
    parity ^= 1u;
    for (uint32_t j = 0; j < NL; ++j)
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                   ::"l"(out + ((size_t)j * p.out_cap + row) * W), "r"(buf + j * W), "r"(W)
                   : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    have = next_hit(row, slot);
    if (have) {
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // the buffer is read
      load(slot);
    }
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // every store has landed
  span_close(p.span);
  if (p.signal) {  // per-layer signal: the hit rows of these layers are one contribution
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
    if (last_block(&g.gather_done[p.layer]) && threadIdx.x == 0)
      for (uint32_t j = p.layer; j < p.layer + NL; ++j) layer_contrib(g, j, 2u, p.round);
  }
}

// ------------------------------------------------------------- exact LRU
//
// Exact LRU's victims beyond the free slots (§3 "PB-LRU", first paragraph: a
// timestamp per slot, victims found by scanning the whole pool): the Q = M - F
// occupied slots with the smallest (timestamp, slot) among those not accessed
// in this round, in that order, written to victims[F + rank].  One cooperative
// launch of co-resident blocks; its phases are separated by grid-wide barriers:
//   1. scan: oldest and newest candidate timestamp, number of candidates;
//   2. radix select on key = timestamp - oldest, 11-bit digits from the top:
//      the threshold timestamp T, and how many slots stamped T are taken (the
//      lowest ones);
//   3. stable compaction, in slot order, of the chosen slots;
//   4. stable LSD radix sort of the chosen (key, slot) pairs on the key's 8-bit
//      digits; the last pass writes the victims.

constexpr unsigned long long kBarrierNs = 1000000000ull;  // a barrier wait gives up after 1 s
constexpr int kLruRegChunks = 4;  // chunks of 4 * kLruThreads stamps a block keeps in registers
constexpr int kLruColLoads = 5;   // per-block counts a lane loads at once (5 * 32 >= 152 blocks)

__device__ __forceinline__ uint32_t ld_acquire(const void *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of a cooperative launch (all blocks co-resident).  Bounded:
// a block that has waited kBarrierNs latches ULA_ERR_TIMEOUT; a block that sees
// an error latched stops waiting.  Returns false (in every thread of the block)
// when the grid must give up.  skip (test hook): this block does not arrive.
__device__ __forceinline__ bool grid_sync(uint32_t *bar, int *status, bool skip = false) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const uint32_t gen = ld_acquire(&bar[1]);
    __threadfence();
    if (skip) {
      ok = 0;
    } else if (atomicAdd(&bar[0], 1u) == gridDim.x - 1) {
      atomicExch(&bar[0], 0u);
      __threadfence();
      atomicAdd(&bar[1], 1u);
    } else {
      const unsigned long long t0 = global_ns();
      uint32_t spins = 0;
      while (ld_acquire(&bar[1]) == gen) {
        if (ld_acquire(status) != 0) {
          ok = 0;
          break;
        }
        if (global_ns() - t0 > kBarrierNs) {
          latch(status, ULA_ERR_TIMEOUT);
          ok = 0;
          break;
        }
        if (++spins > 256) __nanosleep(128);  // poll tightly at first
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

template <typename Op>
__device__ __forceinline__ uint32_t block_reduce(uint32_t v, Op op, uint32_t ident) {
  __shared__ uint32_t ws[kLruThreads / 32];
  __shared__ uint32_t res;
#pragma unroll
  for (int d = 16; d; d >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, d));
  if (lane_id() == 0) ws[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t x = threadIdx.x < kLruThreads / 32 ? ws[threadIdx.x] : ident;
#pragma unroll
    for (int d = 16; d; d >>= 1) x = op(x, __shfl_xor_sync(0xffffffffu, x, d));
    if (threadIdx.x == 0) res = x;
  }
  __syncthreads();
  const uint32_t r = res;
  __syncthreads();
  return r;
}

struct OpMin {
  __device__ uint32_t operator()(uint32_t a, uint32_t b) const { return a < b ? a : b; }
};
struct OpMax {
  __device__ uint32_t operator()(uint32_t a, uint32_t b) const { return a > b ? a : b; }
};
struct OpAdd {
  __device__ uint32_t operator()(uint32_t a, uint32_t b) const { return a + b; }
};

// Four consecutive stamps [i, i+4) (i a multiple of 4); those at or past `end` read
// as kNone (never a candidate).
__device__ __forceinline__ uint4 load4(const uint32_t *stamp, uint32_t i, uint32_t end) {
  if (i + 4 <= end) return __ldcg(reinterpret_cast<const uint4 *>(stamp + i));
  uint4 v = make_uint4(kNone, kNone, kNone, kNone);
  if (i < end) v.x = __ldcg(stamp + i);
  if (i + 1 < end) v.y = __ldcg(stamp + i + 1);
  if (i + 2 < end) v.z = __ldcg(stamp + i + 2);
  return v;
}

// Shared memory of the exact-LRU kernel.
struct LruSmem {
  uint32_t hist[kLruBins];
  uint32_t wcnt[kLruThreads / 32][kSortBins];
  uint32_t off[kSortBins];
  uint32_t pick[2];
};

// The general path: the exact oldest timestamp first (a scan), then a radix select
// over all 32 bits of key = stamp - oldest, a stable compaction and a stable LSD
// sort.  Returns the threshold timestamp T, or kNone when the grid gives up.
__device__ uint32_t lru_general(const LruParams &p, LruSmem &sm, uint32_t Q, uint32_t F) {
  uint32_t *s_hist = sm.hist;
  uint32_t(*s_wcnt)[kSortBins] = sm.wcnt;
  uint32_t *s_off = sm.off;
  uint32_t *s_pick = sm.pick;
  const GroupDev &g = p.grp;
  const uint32_t r = p.round, S = p.geo.S;
  const uint32_t G = gridDim.x, b = blockIdx.x, t = threadIdx.x;
  const uint32_t tid = b * kLruThreads + t, nthr = G * kLruThreads;
  const uint32_t *stamp = g.stamp;
  const uint32_t S4 = (S + 3) / 4;  // groups of four stamps
  uint32_t *victims = g.victims;
  const LruScratch &sc = p.sc;

  // ---- 1. oldest / newest candidate timestamp and the candidates' count.
  // A candidate is an occupied slot not accessed in this round (stamp < r; a
  // free slot's stamp is kNone).
  uint32_t lo = kNone, hi = 0, cnt = 0;
  for (uint32_t q = tid; q < S4; q += nthr) {
    const uint4 v = load4(stamp, 4 * q, S);
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (x[j] < r) {
        lo = min(lo, x[j]);
        hi = max(hi, x[j]);
        ++cnt;
      }
  }
  lo = block_reduce(lo, OpMin(), kNone);
  hi = block_reduce(hi, OpMax(), 0u);
  cnt = block_reduce(cnt, OpAdd(), 0u);
  if (t == 0) sc.blk[b] = make_uint4(lo, hi, cnt, 0);
  for (uint32_t i = tid; i < kLruSelectPasses * kLruBins; i += nthr) sc.hist[i] = 0;
  if (!grid_sync(sc.bar, p.status)) return kNone;
  lo = kNone;
  hi = 0;
  cnt = 0;
  for (uint32_t j = t; j < G; j += kLruThreads) {
    const uint4 v = __ldcg(&sc.blk[j]);
    lo = min(lo, v.x);
    hi = max(hi, v.y);
    cnt += v.z;
  }
  lo = block_reduce(lo, OpMin(), kNone);
  hi = block_reduce(hi, OpMax(), 0u);
  cnt = block_reduce(cnt, OpAdd(), 0u);
  if (cnt < Q) {  // the capacity check rules this out (same values in every block)
    if (b == 0 && t == 0) latch(p.status, ULA_ERR_INTERNAL);
    return kNone;
  }

  // ---- 2. radix select: the Q-th smallest key, digit by digit from the top
  const uint32_t span = hi - lo;
  const int nbits = span ? 32 - __clz(span) : 0;
  uint32_t prefix = 0, rem = Q;  // rem: how many still to take at or above the prefix
  int done = 0;
  for (int pass = 0; done < nbits; ++pass) {
    const int width = min(kLruDigit, nbits - done);
    const int shift = nbits - done - width;
    const uint32_t nb = 1u << width, mask = nb - 1;
    for (uint32_t i = t; i < nb; i += kLruThreads) s_hist[i] = 0;
    __syncthreads();
    for (uint32_t q = tid; q < S4; q += nthr) {
      const uint4 v = load4(stamp, 4 * q, S);
      const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (x[j] < r) {
          const uint32_t key = x[j] - lo;
          if (((unsigned long long)key >> (shift + width)) == prefix)
            atomicAdd(&s_hist[(key >> shift) & mask], 1u);
        }
    }
    __syncthreads();
    uint32_t *gh = sc.hist + (size_t)pass * kLruBins;
    for (uint32_t i = t; i < nb; i += kLruThreads)
      if (s_hist[i]) atomicAdd(&gh[i], s_hist[i]);
    if (!grid_sync(sc.bar, p.status)) return kNone;
    // every block finds the same digit: the first whose running count reaches rem
    uint32_t c4[4], sum = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t bin = 4 * t + j;
      c4[j] = bin < nb ? __ldcg(&gh[bin]) : 0u;
      sum += c4[j];
    }
    uint32_t tot;
    const uint32_t excl = block_incl_scan<kLruThreads>(sum, &tot) - sum;
    if (tot < rem) {
      if (b == 0 && t == 0) latch(p.status, ULA_ERR_INTERNAL);
      return kNone;
    }
    if (excl < rem && rem <= excl + sum) {
      uint32_t acc = excl;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (acc + c4[j] >= rem) {
          s_pick[0] = 4 * t + j;
          s_pick[1] = acc;
          break;
        }
        acc += c4[j];
      }
    }
    __syncthreads();
    prefix = (prefix << width) | s_pick[0];
    rem -= s_pick[1];
    done += width;
    __syncthreads();
  }
  const uint32_t T = lo + prefix;  // threshold timestamp
  const uint32_t need = rem;       // slots stamped T that are taken, lowest first

  // ---- 3. stable compaction in slot order: stamp < T, or stamp == T among the
  // first `need` such slots.  Block b owns slots [s0, s1), four per thread per chunk.
  const uint32_t per = (((S + G - 1) / G) + 3) & ~3u;
  const uint32_t s0 = min(S, b * per), s1 = min(S, s0 + per);
  uint32_t n_lt = 0, n_eq = 0;
  for (uint32_t base = s0; base < s1; base += 4 * kLruThreads) {
    const uint4 v = load4(stamp, base + 4 * t, s1);
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      n_lt += x[j] < T;
      n_eq += x[j] == T;
    }
  }
  n_lt = block_reduce(n_lt, OpAdd(), 0u);
  n_eq = block_reduce(n_eq, OpAdd(), 0u);
  if (t == 0) sc.blk[G + b] = make_uint4(n_lt, n_eq, 0, 0);  // (phase 1 used blk[0, G))
  if (!grid_sync(sc.bar, p.status)) return kNone;
  uint32_t run_lt = 0, run_eq = 0;  // slots below / at the threshold before this block
  for (uint32_t j = t; j < b; j += kLruThreads) {
    const uint4 v = __ldcg(&sc.blk[G + j]);
    run_lt += v.x;
    run_eq += v.y;
  }
  run_lt = block_reduce(run_lt, OpAdd(), 0u);
  run_eq = block_reduce(run_eq, OpAdd(), 0u);
  for (uint32_t base = s0; base < s1; base += 4 * kLruThreads) {
    const uint32_t i = base + 4 * t;
    const uint4 v = load4(stamp, i, s1);
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
    uint32_t mine = 0;  // (below << 16) | at, this thread's four slots
#pragma unroll
    for (int j = 0; j < 4; ++j) mine += ((x[j] < T) << 16) | (x[j] == T);
    uint32_t tot;
    uint32_t before = block_incl_scan<kLruThreads>(mine, &tot) - mine;
    uint32_t lt_before = run_lt + (before >> 16), eq_before = run_eq + (before & 0xffffu);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool is_lt = x[j] < T, is_eq = x[j] == T;
      if (is_lt || (is_eq && eq_before < need)) {
        const uint32_t pos = lt_before + min(eq_before, need);
        if (pos < Q) sc.list[0][pos] = make_uint2(x[j] - lo, i + j);
        else latch(p.status, ULA_ERR_INTERNAL);
      }
      lt_before += is_lt;
      eq_before += is_eq;
    }
    run_lt += tot >> 16;
    run_eq += tot & 0xffffu;
  }
  if (!grid_sync(sc.bar, p.status)) return kNone;

  // ---- 4. order the chosen slots by (timestamp, slot): the list is in slot
  // order, so a stable sort on the key is enough
  const uint32_t kmax = T - lo;
  const int sbits = kmax ? 32 - __clz(kmax) : 0;
  const int spasses = (sbits + 7) / 8;
  if (spasses == 0) {  // one timestamp: slot order is the order
    for (uint32_t i = tid; i < Q; i += nthr) victims[F + i] = __ldcg(&sc.list[0][i]).y;
    return T;
  }
  const uint32_t chunk = (Q + G - 1) / G;
  const uint32_t c0 = min(Q, b * chunk), c1 = min(Q, c0 + chunk);
  const uint32_t warp = t >> 5, lane = lane_id();
  uint2 *src = sc.list[0], *dst = sc.list[1];
  for (int ps = 0; ps < spasses; ++ps) {
    const int shift = 8 * ps;
    const bool last = ps == spasses - 1;
    // (a) this block's digit counts, stored digit-major: table[d][b]
    for (uint32_t i = t; i < kSortBins; i += kLruThreads) s_hist[i] = 0;
    __syncthreads();
    for (uint32_t i = c0 + t; i < c1; i += kLruThreads)
      atomicAdd(&s_hist[(__ldcg(&src[i]).x >> shift) & 0xffu], 1u);
    __syncthreads();
    for (uint32_t d = t; d < kSortBins; d += kLruThreads) sc.table[(size_t)d * G + b] = s_hist[d];
    if (!grid_sync(sc.bar, p.status)) return kNone;
    // (b) per digit (blocks take digits in turn): exclusive prefix over blocks in
    // place; the digit's total goes to table[256 * G + d]
    for (uint32_t d = b; d < kSortBins; d += G) {
      uint32_t *col = sc.table + (size_t)d * G;
      uint32_t run = 0;
      for (uint32_t j0 = 0; j0 < G; j0 += kLruThreads) {
        const uint32_t j = j0 + t;
        const uint32_t v = j < G ? __ldcg(&col[j]) : 0u;
        uint32_t tot;
        const uint32_t inc = block_incl_scan<kLruThreads>(v, &tot);
        if (j < G) col[j] = run + inc - v;
        run += tot;
      }
      if (t == 0) sc.table[(size_t)kSortBins * G + d] = run;
    }
    if (!grid_sync(sc.bar, p.status)) return kNone;
    // (c) this block's start for each digit
    {
      const uint32_t v = t < kSortBins ? __ldcg(&sc.table[(size_t)kSortBins * G + t]) : 0u;
      uint32_t tot;
      const uint32_t inc = block_incl_scan<kLruThreads>(v, &tot);
      if (t < kSortBins) s_off[t] = inc - v + __ldcg(&sc.table[(size_t)t * G + b]);
    }
    __syncthreads();
    // (d) stable scatter, a tile of kLruThreads elements at a time
    for (uint32_t base = c0; base < c1; base += kLruThreads) {
      const uint32_t i = base + t;
      const bool valid = i < c1;
      uint2 e = make_uint2(0, 0);
      uint32_t d = kSortBins;  // invalid lanes form their own group
      if (valid) {
        e = __ldcg(&src[i]);
        d = (e.x >> shift) & 0xffu;
      }
      for (uint32_t k = t; k < (kLruThreads / 32) * kSortBins; k += kLruThreads)
        (&s_wcnt[0][0])[k] = 0;
      __syncthreads();
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      const uint32_t lrank = __popc(peers & ((1u << lane) - 1u));
      if (valid && lrank == 0) s_wcnt[warp][d] = __popc(peers);
      __syncthreads();
      if (valid) {
        uint32_t rank = s_off[d] + lrank;
        for (uint32_t w = 0; w < warp; ++w) rank += s_wcnt[w][d];
        if (rank >= Q) latch(p.status, ULA_ERR_INTERNAL);
        else if (last) victims[F + rank] = e.y;
        else dst[rank] = e;
      }
      __syncthreads();
      if (t < kSortBins) {
        uint32_t add = 0;
        for (uint32_t w = 0; w < kLruThreads / 32; ++w) add += s_wcnt[w][t];
        s_off[t] += add;
      }
      __syncthreads();
    }
    if (last) break;
    if (!grid_sync(sc.bar, p.status)) return kNone;
    uint2 *tmp = src;
    src = dst;
    dst = tmp;
  }
  return T;
}

// (512 threads at <= 64 registers: it fits on an SM beside the gathers.)
//
// The fast path, taken when the Q oldest candidates are stamped within the
// window [lo, lo + nb - 2] of nb <= kLruBins rounds, lo being a lower bound of
// every candidate's stamp kept from the previous scan (the threshold T of a scan
// bounds the stamps left: every older one was chosen and refilled, and stamps
// only grow).  One grid-wide barrier:
//   A. every block histograms key = min(stamp - lo, nb - 1) over its own
//      contiguous slot range (kept in shared memory), publishes the row and adds
//      it to the pool's totals;
//   C. every block: running totals, the first key dT whose running total reaches
//      Q (T = lo + dT) and how many slots stamped T are taken (need); then, for
//      keys <= dT, how many slots of each lie in earlier blocks;
//   D. every block that holds chosen slots lists them in slot order;
//   E. one warp per block ranks them: rank = (candidates with a smaller key) +
//      (same key in earlier blocks) + (same key earlier in this block).
// The totals are accumulated in one of two buffers while the other is cleared
// for the next launch.  Otherwise the general path (lru_general) runs.
__global__ void __launch_bounds__(kLruThreads, 2) k_lru_select(LruParams p) {
  __shared__ LruSmem sm;
  __shared__ uint32_t s_own[kLruBins];  // this block's histogram
  if (ld_acquire(p.status) != 0) return;
  const GroupDev &g = p.grp;
  const uint32_t M = __ldcg(&g.cnt->M), F = __ldcg(&g.cnt->F);
  if (M <= F) return;  // no occupied slot is needed
  const uint32_t Q = M - F, r = p.round, S = p.geo.S;
  const uint32_t G = gridDim.x, b = blockIdx.x, t = threadIdx.x;
  const uint32_t lane = lane_id(), warp = t >> 5;
  const uint32_t *stamp = g.stamp;
  const LruScratch &sc = p.sc;
  const uint32_t lo = __ldcg(&g.cnt->lru_lo);
  const uint32_t par = ld_acquire(&sc.bar[2]) & 1u;
  uint32_t *totals = sc.totals + par * kLruBins;
  const uint32_t per = sc.per;
  const uint32_t s0 = min(S, b * per), s1 = min(S, s0 + per);
  // keys 0 .. r-1-lo; nb bins, the last one also collecting every older-than-window key
  const uint32_t span = r - lo;  // >= 1 (lo <= every candidate's stamp < r)
  uint32_t nb = kLruBins;
  if (span < kLruBins) {
    nb = 2;
    while (nb <= span) nb <<= 1;
  }

  // ---- A. the block's histogram.  When the block's range fits in kLruRegChunks
  // chunks (the same for every block), its stamps are loaded once, all at once, and
  // kept in registers for phase D.
  const bool in_regs = per <= kLruRegChunks * 4 * kLruThreads;
  uint4 sv[kLruRegChunks];
  if (in_regs) {
#pragma unroll
    for (int c = 0; c < kLruRegChunks; ++c) sv[c] = load4(stamp, s0 + (c * kLruThreads + t) * 4, s1);
  }
  for (uint32_t k = t; k < nb; k += kLruThreads) s_own[k] = 0;
  __syncthreads();
  bool bad = false;
  auto hist4 = [&](const uint4 v) {
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool cand = x[j] < r;
      bad |= cand && x[j] < lo;
      const uint32_t key = cand ? min(x[j] - lo, nb - 1) : kNone;
      const uint32_t peers = __match_any_sync(0xffffffffu, key);
      if (cand && lane == (uint32_t)(__ffs(peers) - 1)) atomicAdd(&s_own[key], __popc(peers));
    }
  };
  if (in_regs) {
#pragma unroll
    for (int c = 0; c < kLruRegChunks; ++c) hist4(sv[c]);
  } else {
    for (uint32_t base = s0; base < s1; base += 4 * kLruThreads) hist4(load4(stamp, base + 4 * t, s1));
  }
  if (bad) latch(p.status, ULA_ERR_INTERNAL);  // a stamp below the bound: the grid gives up
  __syncthreads();
  uint32_t *row = sc.rows + (size_t)b * kLruBins;
  for (uint32_t k = t; k < nb; k += kLruThreads) {
    const uint32_t v = s_own[k];
    row[k] = v;
    if (v) atomicAdd(&totals[k], v);
  }
  uint32_t *other = sc.totals + (par ^ 1u) * kLruBins;  // cleared for the next launch
  for (uint32_t k = b * kLruThreads + t; k < kLruBins; k += G * kLruThreads) other[k] = 0;
  if (!grid_sync(sc.bar, p.status, p.stall && b == 0)) return;
  if (b == 0 && t == 0) atomicXor(&sc.bar[2], 1u);  // every block has read the parity

  // ---- C. running totals (sm.hist[k]: candidates with a key below k) and the threshold
  uint32_t c4[4], sum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t k = 4 * t + j;
    c4[j] = k < nb ? __ldcg(&totals[k]) : 0u;
    sum += c4[j];
  }
  uint32_t tot;
  const uint32_t excl = block_incl_scan<kLruThreads>(sum, &tot) - sum;
  {
    uint32_t acc = excl;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sm.hist[4 * t + j] = acc;
      if (acc < Q && Q <= acc + c4[j]) {
        sm.pick[0] = 4 * t + j;
        sm.pick[1] = acc;
      }
      acc += c4[j];
    }
  }
  __syncthreads();
  if (tot < Q) {  // the capacity check rules this out (same in every block)
    if (b == 0 && t == 0) latch(p.status, ULA_ERR_INTERNAL);
    return;
  }
  uint32_t T;
  if (sm.hist[nb - 1] < Q) {  // the window holds fewer than Q candidates
    T = lru_general(p, sm, Q, F);
  } else {
    const uint32_t dT = sm.pick[0], need = Q - sm.pick[1];
    // slots of each key <= dT in earlier blocks (sm.off is too small for many keys:
    // use the per-warp table's storage, kLruThreads/32 * kSortBins >= kLruBins words)
    uint32_t *pre = &sm.wcnt[0][0];
    for (uint32_t k = warp; k <= dT; k += kLruThreads / 32) {
      uint32_t acc = 0;
      for (uint32_t j0 = 0; j0 < b; j0 += 32 * kLruColLoads) {
        uint32_t v[kLruColLoads];
#pragma unroll
        for (int u = 0; u < kLruColLoads; ++u) {
          const uint32_t j = j0 + 32 * u + lane;
          v[u] = j < b ? __ldcg(&sc.rows[(size_t)j * kLruBins + k]) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kLruColLoads; ++u) acc += v[u];
      }
      acc = warp_sum(acc);
      if (lane == 0) pre[k] = acc;
    }
    __syncthreads();
    const uint32_t eq_prefix = pre[dT];
    const uint32_t cap = need > eq_prefix ? need - eq_prefix : 0u;
    uint32_t mine_lt = 0;
    for (uint32_t k = t; k < dT; k += kLruThreads) mine_lt += s_own[k];
    const uint32_t n_b = block_reduce(mine_lt, OpAdd(), 0u) + min(s_own[dT], cap);

    if (n_b) {
      // ---- D. the block's chosen slots in slot order: key < dT, or key == dT
      // within the first `need` of the pool (eq_prefix of them lie in earlier blocks)
      uint2 *blist = sc.blist + (size_t)b * per;
      auto take = [&](const uint32_t i, const uint32_t *key, uint32_t lt_b, uint32_t eq_b) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool is_lt = key[j] < dT, is_eq = key[j] == dT;
          if (is_lt || (is_eq && eq_b < cap)) {
            const uint32_t pos = lt_b + min(eq_b, cap);
            if (pos < per) blist[pos] = make_uint2(key[j], i + j);
            else latch(p.status, ULA_ERR_INTERNAL);
          }
          lt_b += is_lt;
          eq_b += is_eq;
        }
      };
      auto keys4 = [&](const uint4 v, uint32_t *key) {
        const uint32_t x[4] = {v.x, v.y, v.z, v.w};
        uint32_t m = 0;  // (below << 16) | at
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          key[j] = x[j] < r ? min(x[j] - lo, nb - 1) : kNone;
          m += ((uint32_t)(key[j] < dT) << 16) | (uint32_t)(key[j] == dT);
        }
        return m;
      };
      if (in_regs) {
        // Piece (c, w) = the 128 slots warp w holds of chunk c; pieces in slot order
        // are c-major.  Warp-level counts, one table of piece totals, one barrier.
        uint32_t *ptot = sm.off;  // [kLruRegChunks * 16] packed piece totals
        uint32_t key[kLruRegChunks][4], incl[kLruRegChunks], mine[kLruRegChunks];
#pragma unroll
        for (int c = 0; c < kLruRegChunks; ++c) {
          mine[c] = keys4(sv[c], key[c]);
          incl[c] = warp_incl_scan(mine[c]);
          if (lane == 31) ptot[c * (kLruThreads / 32) + warp] = incl[c];
        }
        __syncthreads();
        // exclusive prefix of all pieces: lane l holds pieces 2l and 2l + 1
        const uint32_t a0 = ptot[2 * lane], a1 = ptot[2 * lane + 1];
        const uint32_t pin = warp_incl_scan(a0 + a1);
#pragma unroll
        for (int c = 0; c < kLruRegChunks; ++c) {
          const uint32_t pc = c * (kLruThreads / 32) + warp;  // this warp's piece
          const uint32_t owner = __shfl_sync(0xffffffffu, pin - a0 - a1, pc >> 1);
          const uint32_t a_even = __shfl_sync(0xffffffffu, a0, pc >> 1);
          const uint32_t pbase = owner + ((pc & 1u) ? a_even : 0u);
          const uint32_t before = pbase + incl[c] - mine[c];
          take(s0 + (c * kLruThreads + t) * 4, key[c], before >> 16, before & 0xffffu);
        }
      } else {
        uint32_t run_lt = 0, run_eq = 0;
        for (uint32_t base = s0; base < s1; base += 4 * kLruThreads) {
          uint32_t key[4];
          const uint32_t m = keys4(load4(stamp, base + 4 * t, s1), key);
          uint32_t ctot;
          const uint32_t before = block_incl_scan<kLruThreads>(m, &ctot) - m;
          take(base + 4 * t, key, run_lt + (before >> 16), run_eq + (before & 0xffffu));
          run_lt += ctot >> 16;
          run_eq += ctot & 0xffffu;
        }
      }

      // ---- E. ranks; sm.hist[k] becomes the first rank of key k in this block
      for (uint32_t k = t; k <= dT; k += kLruThreads) sm.hist[k] += pre[k];
      __syncthreads();
      if (dT < kSortBins) {  // tiles of kLruThreads list entries, per-warp key counts
        uint32_t(*wc)[kSortBins] = sm.wcnt;  // (pre is no longer needed)
        for (uint32_t i0 = 0; i0 < n_b; i0 += kLruThreads) {
          const uint32_t i = i0 + t;
          const bool valid = i < n_b;
          const uint2 e = valid ? blist[i] : make_uint2(kSortBins, 0u);
          for (uint32_t k = t; k < (kLruThreads / 32) * (dT + 1); k += kLruThreads)
            wc[k / (dT + 1)][k % (dT + 1)] = 0;
          __syncthreads();
          const uint32_t peers = __match_any_sync(0xffffffffu, e.x);
          const uint32_t lrank = __popc(peers & ((1u << lane) - 1u));
          if (valid && lrank == 0) wc[warp][e.x] = __popc(peers);
          __syncthreads();
          if (valid) {
            uint32_t rank = sm.hist[e.x] + lrank;
            for (uint32_t w = 0; w < warp; ++w) rank += wc[w][e.x];
            if (rank < Q) g.victims[F + rank] = e.y;
            else latch(p.status, ULA_ERR_INTERNAL);
          }
          __syncthreads();
          for (uint32_t k = t; k <= dT; k += kLruThreads) {
            uint32_t add = 0;
            for (uint32_t w = 0; w < kLruThreads / 32; ++w) add += wc[w][k];
            sm.hist[k] += add;
          }
          __syncthreads();
        }
      } else if (warp == 0) {  // many keys: one warp, in order
        for (uint32_t i0 = 0; i0 < n_b; i0 += 32) {
          const uint32_t i = i0 + lane;
          const bool valid = i < n_b;
          const uint2 e = valid ? blist[i] : make_uint2(kNone, 0u);
          const uint32_t peers = __match_any_sync(0xffffffffu, e.x);
          const uint32_t lrank = __popc(peers & ((1u << lane) - 1u));
          const uint32_t rank = valid ? sm.hist[e.x] + lrank : 0u;
          __syncwarp();
          if (valid && lrank == 0) sm.hist[e.x] += __popc(peers);
          __syncwarp();
          if (valid) {
            if (rank < Q) g.victims[F + rank] = e.y;
            else latch(p.status, ULA_ERR_INTERNAL);
          }
        }
      }
    }
    T = lo + dT;
  }
  // the threshold bounds every stamp left for the next scan
  if (T != kNone && b == 0 && t == 0) g.cnt->lru_lo = T;
}

// ------------------------------------------------------------ alloc / free

// Alloc, per group (one block each): walk the free class for n slots, then the
// host-free bitmap for the rest.
__global__ void __launch_bounds__(kScanThreads) k_alloc_select(EmitParams p) {
  if (block_skips(p.status)) return;
  const GroupDev g = p.groups[p.group0 + blockIdx.x];
  select_walk<kScanThreads>(g, p.geo, p.order, p.quota, p.quota, false, p.status);
}

// Alloc: address i of the range goes to the i-th selected free GPU slot (the
// lowest ones, joining the current bucket), the rest to the selected host slots.
__global__ void __launch_bounds__(256) k_alloc_place(AllocParams p) {
  if (*(volatile int *)p.status) return;
  const uint32_t gi = p.group0 + blockIdx.y;
  const GroupDev g = p.groups[gi];
  const Geometry &geo = p.geo;
  const uint32_t F = g.cnt->F;
  const uint32_t lane = lane_id();
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
  const size_t sb = (size_t)g.layers * geo.W;
  const uint32_t nvec = (uint32_t)(sb / 16);
  const uint32_t round = p.round[gi], cur = round % geo.B;
  for (uint32_t i = warp; i < p.n; i += nwarps) {
    const uint32_t a = p.base + i;
    const bool on_gpu = i < F;
    const uint32_t slot = on_gpu ? g.victims[i] : g.wb_host[i - F];
    if ((on_gpu && slot >= geo.S) || (!on_gpu && slot >= geo.H) || a >= geo.max_logical) {
      if (lane == 0) latch(p.status, ULA_ERR_INTERNAL);
      continue;
    }
    const uint4 *src =
        reinterpret_cast<const uint4 *>(p.rows + p.group_off[gi] + (size_t)i * p.row_stride * sb);
    uint4 *dst = reinterpret_cast<uint4 *>((on_gpu ? g.gpu_pool : g.host_pool) + (size_t)slot * sb);
    for (uint32_t c = lane; c < nvec; c += 32) dst[c] = src[c];
    __syncwarp();
    if (lane == 0) {
      if (on_gpu) {
        g.map[a] = slot;
        g.owner[slot] = a;
        g.stamp[slot] = round;
        bm_clear(class_bitmap(g, geo, geo.B + 1), slot);
        bm_set(class_bitmap(g, geo, access_class(geo, cur)), slot);
      } else {
        g.map[a] = kHostBit | slot;
      }
    }
  }
}

// Free: every address's slot is released (GPU: leaves its class, joins free).
__global__ void k_free(FreeParams p) {
  if (*(volatile int *)p.status) return;
  const uint32_t gi = p.group0 + blockIdx.y;
  const GroupDev g = p.groups[gi];
  const Geometry &geo = p.geo;
  const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= p.n) return;
  const uint32_t a = p.base + i;
  const uint32_t m = g.map[a];
  if (m == kUnalloc) {  // (a local buffer need not hold every address it drops)
    if (!geo.cache) latch(p.status, ULA_ERR_INTERNAL);
    return;
  }
  if (m & kHostBit) {
    const uint32_t hs = m & kSlotMask;
    if (hs >= geo.H) {
      latch(p.status, ULA_ERR_INTERNAL);
      return;
    }
    bm_set(host_free_bitmap(g), hs);
    atomicAdd(&g.cnt->free_host, 1u);
  } else {
    if (m >= geo.S) {
      latch(p.status, ULA_ERR_INTERNAL);
      return;
    }
    const uint32_t c = slot_class(geo, g.stamp[m], p.round[gi]);
    if (c == geo.B + 1) {
      latch(p.status, ULA_ERR_INTERNAL);
      return;
    }
    bm_clear(class_bitmap(g, geo, c), m);
    bm_set(class_bitmap(g, geo, geo.B + 1), m);
    g.stamp[m] = kNone;
    g.owner[m] = kNone;
    atomicAdd(&g.cnt->free_gpu, 1u);
  }
  g.map[a] = kUnalloc;
}

// TP mode: each entry as every partition and every rank's buffer sees it.
__global__ void k_tp_split(const uint32_t *sel, uint32_t E, uint32_t P, uint32_t *part_sel,
                           uint32_t *buf_sel, uint32_t stride) {
  const uint32_t e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const uint32_t a = sel[e];
  const uint32_t own = a == kPad ? kNone : a % P;
  for (uint32_t p = 0; p < P; ++p) {
    part_sel[(size_t)p * stride + e] = own == p ? a / P : kPad;
    buf_sel[(size_t)p * stride + e] = (own == kNone || own == p) ? kPad : a;
  }
}

// A model consumer of one layer: one block polls the layer's flag (acquire) until
// it holds the round, bounded by kBarrierNs, then sums the layer's rows.
__global__ void k_consume(const uint32_t *flag, uint32_t round, const uint8_t *out,
                          uint32_t out_cap, uint32_t layer, uint32_t n_rows, uint32_t W,
                          unsigned long long *result) {
  __shared__ int s_ok;
  __shared__ unsigned long long s_seen;
  if (threadIdx.x == 0) {
    const unsigned long long t0 = global_ns();
    int ok = 1;
    while (ld_acquire(flag) != round) {
      if (global_ns() - t0 > kBarrierNs) {
        ok = 0;
        break;
      }
    }
    s_ok = ok;
    s_seen = global_ns();
  }
  __syncthreads();
  if (!s_ok) {
    if (threadIdx.x == 0) {
      result[0] = s_seen;
      result[1] = 0;
      result[2] = ULA_ERR_TIMEOUT;
    }
    return;
  }
  const uint32_t *words = reinterpret_cast<const uint32_t *>(out + (size_t)layer * out_cap * W);
  const size_t n = (size_t)n_rows * W / 4;
  uint32_t sum = 0;
  for (size_t i = threadIdx.x; i < n; i += blockDim.x) sum += __ldcg(&words[i]);
  sum = warp_sum(sum);
  __shared__ uint32_t ws[32];
  if (lane_id() == 0) ws[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t tot = 0;
    for (uint32_t w = 0; w < blockDim.x / 32; ++w) tot += ws[w];
    result[0] = s_seen;
    result[1] = tot;
    result[2] = 0;
  }
}

inline uint32_t div_up(uint64_t a, uint64_t b) { return (uint32_t)((a + b - 1) / b); }

// A launch that may start while the previous kernel on the stream finishes (the
// kernel calls pdl_wait() before it reads anything that kernel wrote).
template <typename P>
cudaError_t launch_dependent(void (*kernel)(P), dim3 grid, dim3 block, cudaStream_t s, const P &p) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace

// --------------------------------------------------------------- launchers

cudaError_t launch_bitmap_fill(Bitmap b, uint32_t nbits, cudaStream_t s) {
  if (nbits == 0) return cudaSuccess;
  const Dims d = dims_for(nbits);
  k_bitmap_fill<<<div_up(d.n0, 256), 256, 0, s>>>(b, nbits);
  return cudaGetLastError();
}

cudaError_t launch_dedup(const StepParams &p, cudaStream_t s) {
  const uint32_t nblk = div_up(p.E, kEntryThreads);
  if (nblk) k_dedup_stamp<<<div_up(p.E, kStampThreads), kStampThreads, 0, s>>>(p);
  return launch_dependent(k_dedup_count_scan, dim3(nblk ? nblk : 1), dim3(kEntryThreads), s, p);
}

cudaError_t launch_rotate_emit(const StepParams &p, cudaStream_t s) {
  StepParams q = p;
  q.emit_blocks = div_up(p.E, kEntryThreads);
  const uint32_t words = p.geo.gd.n0 > p.geo.gd.n1 ? p.geo.gd.n0 : p.geo.gd.n1;
  uint32_t rot = p.geo.exact ? 0u : div_up(words, kEntryThreads * 4);
  const uint32_t grid = q.emit_blocks + rot;
  return launch_dependent(k_rotate_emit, dim3(grid ? grid : 1), dim3(kEntryThreads), s, q);
}

cudaError_t launch_mark_select(const StepParams &p, cudaStream_t s) {
  // one warp per segment of the class bitmaps (the marking), at least one block (the walk)
  const uint32_t nblk = div_up(p.geo.nseg, kEntryThreads / 32);
  return launch_dependent(k_mark_select, dim3(nblk ? nblk : 1), dim3(kEntryThreads), s, p);
}

cudaError_t launch_select_emit(const EmitParams &p, uint32_t n_groups, int blocks, cudaStream_t s) {
  const uint32_t grid = (uint32_t)(blocks > 0 ? blocks : 1) + (p.fill_order ? 1u : 0u);
  return launch_dependent(k_select_emit, dim3(grid, n_groups), dim3(kOrderThreads), s, p);
}

cudaError_t launch_alloc_select(const EmitParams &p, uint32_t n_groups, cudaStream_t s) {
  k_alloc_select<<<n_groups, kScanThreads, 0, s>>>(p);
  return cudaGetLastError();
}

size_t gather_bulk_smem(uint32_t slot_bytes) {
  return kBulkBars + (size_t)kBulkThreads * slot_bytes;
}

// The bulk gather's shared memory is capped so that at least two of its blocks fit on an
// SM beside the other kernels' blocks.
constexpr size_t kBulkMaxSmem = 100 * 1024;

bool gather_uses_bulk(uint32_t slot_bytes) { return gather_bulk_smem(slot_bytes) <= kBulkMaxSmem; }

cudaError_t resident_blocks(int *move_per_sm, int *gather_per_sm, uint32_t slot_bytes) {
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(move_per_sm, k_move, kMoveThreads, 0);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_gather_bulk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kBulkMaxSmem);
  if (e != cudaSuccess) return e;
  if (gather_uses_bulk(slot_bytes))
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(gather_per_sm, k_gather_bulk, kBulkThreads,
                                                         gather_bulk_smem(slot_bytes));
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(gather_per_sm, k_gather, kGatherThreads, 0);
}

int move_threads() { return kMoveThreads; }

cudaError_t launch_stage(const MoveParams &p, int blocks, cudaStream_t s) {
  // Chained to the hit gather by programmatic dependent launch: it reads nothing the
  // gather writes, so it needs no wait, and it is launched as the gather's last blocks
  // end instead of after the gather's completion (the step about 1 % shorter).  (With
  // the earlier register gather a chained staging copy slowed the move that followed:
  // 246-252 against 295-301 GB/s.)
  return launch_dependent(k_stage, dim3(blocks > 0 ? blocks : 1), dim3(256), s, p);
}

cudaError_t launch_move(const MoveParams &p, int blocks, bool dependent, cudaStream_t s) {
  if (!p.geo.signal) {  // copies, then each victim's map, in one kernel
    if (dependent) return launch_dependent(k_move, dim3(blocks), dim3(kMoveThreads), s, p);
    k_move<<<blocks, kMoveThreads, 0, s>>>(p);
    return cudaGetLastError();
  }
  // layer by layer: a victim's chunks are spread over warps, so the map follows in
  // a second kernel, once every copy is done
  cudaError_t e = launch_dependent(k_move_layers, dim3(blocks), dim3(256), s, p);
  if (e != cudaSuccess) return e;
  return launch_dependent(k_commit, dim3(blocks), dim3(256), s, p);
}

cudaError_t launch_tp_split(const uint32_t *sel, uint32_t E, uint32_t P, uint32_t *part_sel,
                            uint32_t *buf_sel, uint32_t stride, cudaStream_t s) {
  if (E) k_tp_split<<<div_up(E, 256), 256, 0, s>>>(sel, E, P, part_sel, buf_sel, stride);
  return cudaGetLastError();
}

cudaError_t launch_consume(const uint32_t *flag, uint32_t round, const uint8_t *out,
                           uint32_t out_cap, uint32_t layer, uint32_t n_rows, uint32_t W,
                           unsigned long long *result, cudaStream_t s) {
  k_consume<<<1, 256, 0, s>>>(flag, round, out, out_cap, layer, n_rows, W, result);
  return cudaGetLastError();
}

cudaError_t lru_resident_blocks(int *per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, k_lru_select, kLruThreads, 0);
}

cudaError_t launch_lru_select(const LruParams &p, int blocks, cudaStream_t s) {
  LruParams q = p;
  void *args[] = {&q};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(k_lru_select), dim3(blocks),
                                     dim3(kLruThreads), args, 0, s);
}

cudaError_t launch_gather(const GatherParams &p, int blocks, cudaStream_t s) {
  const uint32_t rb = p.nlayers * p.geo.W;
  if (gather_uses_bulk(rb))
    k_gather_bulk<<<blocks, kBulkThreads, gather_bulk_smem(rb), s>>>(p);
  else
    k_gather<<<blocks, kGatherThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_alloc_place(const AllocParams &p, uint32_t n_groups, int max_blocks,
                               cudaStream_t s) {
  uint32_t blocks = div_up((uint64_t)p.n * 32, 256);
  const uint32_t cap = (uint32_t)max_blocks;
  if (blocks > cap) blocks = cap;
  dim3 grid(blocks ? blocks : 1, n_groups);
  k_alloc_place<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_free(const FreeParams &p, uint32_t n_groups, cudaStream_t s) {
  dim3 grid(div_up(p.n, 256) ? div_up(p.n, 256) : 1, n_groups);
  k_free<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ula
