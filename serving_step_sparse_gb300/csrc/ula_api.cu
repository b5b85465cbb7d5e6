// Host orchestrator behind the C ABI (include/ula.h): context set-up, argument
// checks, stream/event ordering, and the per-call kernel sequences.
//
// Ordering rules (UlaCache summary page, §2 on layer groups sharing one selection, and §3
// last paragraph: the data moves first, then the map, then the signal).  A step's metadata
// kernels run on the context's metadata stream, chained by programmatic dependent launch:
// dedup/translate + capacity check -> rotate/compact -> mark/victim walk -> victim emit.
// Its copies run on the copy stream after an event on that metadata: the hit gather (every
// layer, one launch), the staging copy of the victims' rows, the move (write-backs, fills,
// each victim's commit), each chained to the one before by programmatic dependent launch.
// A group's step waits only for that group's previous step (its commit and gather
// events) and its last alloc/free, so one call's metadata runs while earlier calls' copies
// run.  With ULA_FLAG_GATHER_BESIDE_MOVE the gather runs instead on the low-priority side
// stream, released after the compaction, beside the rest.  The caller's stream waits for
// the commit and the gather; alloc/free run per group, on the group's update stream, after
// the group's step in flight.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "ula_device.cuh"

using namespace ula;

namespace {

constexpr uint32_t kAllocChunk = 65536;
#ifndef ULA_CACHE_MOVE_BLOCKS
#define ULA_CACHE_MOVE_BLOCKS 4  // move blocks per SM of a TP rank's local buffer (HBM copies)
#endif
constexpr size_t kSpanCap = 1u << 16;  // span records kept between reads
// Internal: a TP rank's local buffer (misses fetched from the owner partitions,
// evicted copies dropped).  Not accepted by the public ula_create.
constexpr uint32_t kFlagCacheInternal = 1u << 31;

#define ULA_CUDA(call)                      \
  do {                                      \
    cudaError_t e_ = (call);                \
    if (e_ != cudaSuccess) return c->fail(e_); \
  } while (0)

}  // namespace

struct ula_ctx {
  ula_config cfg{};
  int device = 0;
  int sm_count = 0;
  cudaStream_t home = nullptr;  // the caller's stream given at create (alloc/free order)
  // Internal streams.  crit: the steps' metadata kernels, alloc and free, in call order.
  // copy: every step's copy kernels (the hit gather before the move, the staging copy,
  // the move), in call order.  side: the hit gather beside the move.  A step's metadata
  // thus runs while the previous call's copies occupy the SMs and the host link (the
  // calls of different groups are independent: each group has its own state and step
  // scratch).
  cudaStream_t crit = nullptr;  // highest priority
  cudaStream_t copy = nullptr;  // highest priority
  cudaStream_t side = nullptr;  // lowest priority
  cudaEvent_t in_evt = nullptr;
  int move_blocks = 0, gather_blocks = 0;  // persistent grids (resident blocks)
  int gather_fit_per_sm = 0;
  int emit_blocks = 0, stage_blocks = 0;
  bool beside = false;  // the hit gather runs beside the move (else before it)
  Geometry geo{};
  std::vector<GroupDev> groups_h;
  GroupDev *groups_d = nullptr;
  GroupCounters *cnt_d = nullptr;
  // A group's step scratch (its own, so that a group's metadata can run while another
  // group's copies still read theirs) and the events that order its steps.
  struct GroupStep {
    unsigned long long *tbl = nullptr;  // [max_logical] dedup stamps
    uint32_t *addr_row = nullptr;       // [max_logical]
    uint2 *blk = nullptr;
    uint32_t *miss_list = nullptr, *miss_hs = nullptr, *miss_row = nullptr;
    uint32_t *fill_order = nullptr;     // [decision_cap] the move's fill order
    uint32_t *vdone = nullptr;          // [decision_cap] copies done per victim
    uint32_t epoch = 0;
    cudaEvent_t rot_evt = nullptr;      // compaction done (the gather may start)
    cudaEvent_t meta_evt = nullptr;     // victims emitted (the copies may start)
    cudaEvent_t commit_evt = nullptr;   // the step's move committed
    cudaEvent_t hit_evt = nullptr;      // the step's hit gather done
    bool in_flight = false;             // commit_evt/hit_evt mark this group's last step
    // alloc/free of this group run on its own stream, after its last step's copies, so
    // that a later step of one group need not wait for every group's copies
    cudaStream_t upd = nullptr;
    cudaEvent_t upd_evt = nullptr;      // the group's last alloc/free done
    bool upd_pending = false;
  };
  std::vector<GroupStep> steps;
  uint8_t *stage = nullptr;        // [min(max_entries, S)][max L_g][W] staged victim rows
  // launch spans of the copy kernels (diagnostics): a ring of records on the device
  SpanRec *spans_d = nullptr;
  bool span_on = false;
  std::vector<uint32_t> span_meta;  // phase << 16 | group of each record taken
  TpSource tp_src[ULA_MAX_GROUPS] = {};  // TP local buffer: the owner partitions per group
  LruScratch lru{};     // exact LRU's scan scratch (ULA_FLAG_EXACT_LRU only)
  int lru_blocks = 0;   // its cooperative grid
  int *status = nullptr;
  uint32_t decision_cap = 0;
  uint32_t round[ULA_MAX_GROUPS] = {};
  uint32_t next_logical = 0;
  uint64_t live_count = 0;
  std::vector<uint8_t> live;
  int poisoned = 0;
  int inject = 0;
  std::vector<void *> allocations;
  // profiling: launch counts always; event pairs per phase instance when enabled
  struct Timed {
    int phase;
    cudaEvent_t a, b;
  };
  bool prof_on = false;
  std::vector<Timed> prof_pending;
  std::vector<cudaEvent_t> prof_spare;
  uint64_t prof_kernels[ULA_PHASE_COUNT] = {};
  uint64_t prof_timed[ULA_PHASE_COUNT] = {};
  double prof_ms[ULA_PHASE_COUNT] = {};

  int fail(cudaError_t e) {
    (void)e;
    poisoned = ULA_ERR_CUDA;
    return ULA_ERR_CUDA;
  }

  template <typename T>
  cudaError_t alloc(T **p, size_t count) {
    void *q = nullptr;
    cudaError_t e = cudaMalloc(&q, count ? count * sizeof(T) : sizeof(T));
    if (e == cudaSuccess) allocations.push_back(q);
    *p = static_cast<T *>(q);
    return e;
  }

  // the call's work on `crit` starts after everything already on the caller's stream
  cudaError_t enter(cudaStream_t caller) {
    cudaError_t e = cudaEventRecord(in_evt, caller);
    return e != cudaSuccess ? e : cudaStreamWaitEvent(crit, in_evt, 0);
  }

  // alloc/free of group g: on the group's own stream, after everything on the home
  // stream (in_evt, recorded by the caller of this helper) and after the group's last
  // step (its copies and gather) and last alloc/free
  cudaError_t begin_update(uint32_t g) {
    GroupStep &st = steps[g];
    cudaError_t e = cudaStreamWaitEvent(st.upd, in_evt, 0);
    if (e == cudaSuccess && st.in_flight) e = cudaStreamWaitEvent(st.upd, st.commit_evt, 0);
    if (e == cudaSuccess && st.in_flight) e = cudaStreamWaitEvent(st.upd, st.hit_evt, 0);
    return e;
  }
  // ... and the home stream continues after every group's update
  cudaError_t end_updates(cudaStream_t home_s) {
    for (GroupStep &st : steps) {
      cudaError_t e = cudaEventRecord(st.upd_evt, st.upd);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(home_s, st.upd_evt, 0);
      if (e != cudaSuccess) return e;
      st.upd_pending = true;
    }
    return cudaSuccess;
  }

  // the next span record for a launch of `phase` in `group`, or NULL (not recording,
  // or the ring is full)
  SpanRec *take_span(int phase, uint32_t group) {
    if (!span_on || span_meta.size() >= kSpanCap) return nullptr;
    span_meta.push_back(((uint32_t)phase << 16) | group);
    return spans_d + (span_meta.size() - 1);
  }


  cudaError_t take_event(cudaEvent_t *e) {
    if (!prof_spare.empty()) {
      *e = prof_spare.back();
      prof_spare.pop_back();
      return cudaSuccess;
    }
    return cudaEventCreate(e);
  }

  // Runs `launch` (which enqueues `kernels` kernels of `phase` on `s`), bracketed
  // by timing events on `s` when profiling is on.
  template <typename F>
  cudaError_t phase(int ph, cudaStream_t s, uint64_t kernels, F &&launch) {
    Timed t{ph, nullptr, nullptr};
    if (prof_on) {
      cudaError_t e = take_event(&t.a);
      if (e == cudaSuccess) e = take_event(&t.b);
      if (e == cudaSuccess) e = cudaEventRecord(t.a, s);
      if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch();
    if (e != cudaSuccess) return e;
    prof_kernels[ph] += kernels;
    if (prof_on) {
      e = cudaEventRecord(t.b, s);
      if (e != cudaSuccess) return e;
      prof_pending.push_back(t);
    }
    return cudaSuccess;
  }

  cudaError_t ensure_device() {
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return e;
    return cur == device ? cudaSuccess : cudaSetDevice(device);
  }
};

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Persistent grid of the move: one block of 128 threads per SM (the host link is
// saturated by 4 warps on every SM; more warps or fewer SMs move less, measured).
constexpr int kMoveBlocksPerSm = 1;
// The step's hit gather is not persistent: short blocks of kGatherRowsPerBlock entries'
// worth of rows, so that the metadata kernels of later calls (highest priority) get SM
// room as its blocks retire and are done before the move, instead of piling up beside
// it.  Its grid is sized from the entry count (U <= E); blocks past the last row exit at
// once.
constexpr uint32_t kGatherRowsPerBlock = 64;
int gather_step_blocks(uint64_t entries) {
  const uint64_t b = (entries + kGatherRowsPerBlock - 1) / kGatherRowsPerBlock;
  return (int)(b < 1 ? 1 : (b > 65535 ? 65535 : b));
}

// blocks per SM from the environment (or `dflt`), clamped to [1, fit]
int env_blocks(const char *name, int dflt, int fit) {
  int v = dflt;
  if (const char *e = std::getenv(name)) {
    const int x = std::atoi(e);
    if (x > 0) v = x;
  }
  if (v > fit) v = fit;
  return v < 1 ? 1 : v;
}

// device-accessible address of a device or pinned host pointer, or nullptr
void *device_address(const void *p, int device, bool allow_device, bool allow_host) {
  if (!p) return nullptr;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type == cudaMemoryTypeDevice && allow_device && at.device == device)
    return const_cast<void *>(p);
  if (at.type == cudaMemoryTypeManaged && allow_device) return const_cast<void *>(p);
  if (at.type == cudaMemoryTypeHost && allow_host) {
    if (at.devicePointer) return at.devicePointer;  // the queried address, as the device sees it
    void *dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, const_cast<void *>(p), 0) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return dp;
  }
  return nullptr;
}

int validate_config(const ula_config *c) {
  if (!c) return ULA_ERR_INVALID_ARG;
  if (c->row_bytes == 0 || c->row_bytes % 16) return ULA_ERR_INVALID_ARG;
  if (c->n_groups == 0 || c->n_groups > ULA_MAX_GROUPS) return ULA_ERR_INVALID_ARG;
  for (uint32_t g = 0; g < c->n_groups; ++g)
    if (c->layers_per_group[g] == 0 || (uint64_t)c->layers_per_group[g] * c->row_bytes > (1u << 30))
      return ULA_ERR_INVALID_ARG;
  if (c->gpu_slots == 0 || c->gpu_slots > kSlotMask || c->host_slots > kSlotMask)
    return ULA_ERR_INVALID_ARG;
  if (c->ring_buckets == 0 || c->ring_buckets > ULA_MAX_BUCKETS) return ULA_ERR_INVALID_ARG;
  if (c->max_logical == 0 || c->max_logical > kSlotMask) return ULA_ERR_INVALID_ARG;
  if (c->max_entries == 0) return ULA_ERR_INVALID_ARG;
  if ((c->flags & ~(ULA_FLAG_BYPASS_OVERFLOW | ULA_FLAG_EXACT_LRU | ULA_FLAG_LAYER_SIGNAL |
                    ULA_FLAG_GATHER_BESIDE_MOVE)) != 0)
    return ULA_ERR_INVALID_ARG;
  return ULA_OK;
}

void destroy_resources(ula_ctx *c) {
  for (void *p : c->allocations) cudaFree(p);
  c->allocations.clear();
  if (c->side) cudaStreamDestroy(c->side);
  if (c->crit) cudaStreamDestroy(c->crit);
  if (c->copy) cudaStreamDestroy(c->copy);
  if (c->in_evt) cudaEventDestroy(c->in_evt);
  for (auto &st : c->steps) {
    for (cudaEvent_t e : {st.rot_evt, st.meta_evt, st.commit_evt, st.hit_evt, st.upd_evt})
      if (e) cudaEventDestroy(e);
    if (st.upd) cudaStreamDestroy(st.upd);
  }
  for (auto &t : c->prof_pending) {
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  for (cudaEvent_t e : c->prof_spare) cudaEventDestroy(e);
}

int create_impl(ula_ctx *c, void *const *gpu_pools, void *const *host_pools) {
  const ula_config &cfg = c->cfg;
  ULA_CUDA(cudaGetDevice(&c->device));
  ULA_CUDA(cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device));
  const uint32_t G = cfg.n_groups, S = cfg.gpu_slots, H = cfg.host_slots, B = cfg.ring_buckets;

  Geometry &geo = c->geo;
  geo.S = S;
  geo.H = H;
  geo.B = B;
  geo.W = cfg.row_bytes;
  geo.max_logical = cfg.max_logical;
  geo.bypass = (cfg.flags & ULA_FLAG_BYPASS_OVERFLOW) ? 1u : 0u;
  geo.exact = (cfg.flags & ULA_FLAG_EXACT_LRU) ? 1u : 0u;
  geo.signal = (cfg.flags & ULA_FLAG_LAYER_SIGNAL) ? 1u : 0u;
  geo.cache = (cfg.flags & kFlagCacheInternal) ? 1u : 0u;
  geo.gd = dims_for(S);
  geo.hd = dims_for(H);
  geo.nseg = geo.gd.n1;
  geo.hseg = geo.hd.n1;
  {  // fill-order buckets: host slot >> fill_shift < kFillBuckets (a local buffer's miss
     // source is partition << 29 | slot: the top 11 bits)
    uint32_t bits = 0;
    while (bits < 32 && (1ull << bits) < (uint64_t)(geo.cache ? 0xFFFFFFFFu : H)) ++bits;
    const uint32_t bucket_bits = 11;  // 2^11 = kFillBuckets
    geo.fill_shift = bits > bucket_bits ? bits - bucket_bits : 0u;
  }
  c->beside = geo.signal || (cfg.flags & ULA_FLAG_GATHER_BESIDE_MOVE);
  c->decision_cap = cfg.max_entries > kAllocChunk ? cfg.max_entries : kAllocChunk;

  // pools: caller-owned, borrowed
  std::vector<uint8_t *> gp(G), hp(G);
  for (uint32_t g = 0; g < G; ++g) {
    void *d = device_address(gpu_pools ? gpu_pools[g] : nullptr, c->device, true, false);
    if (!d || !aligned16(d)) return ULA_ERR_INVALID_ARG;
    gp[g] = static_cast<uint8_t *>(d);
    if (H) {
      void *h = device_address(host_pools ? host_pools[g] : nullptr, c->device, false, true);
      if (!h || !aligned16(h)) return ULA_ERR_INVALID_ARG;
      hp[g] = static_cast<uint8_t *>(h);
    }
  }

  int prio_least = 0, prio_greatest = 0;
  ULA_CUDA(cudaDeviceGetStreamPriorityRange(&prio_least, &prio_greatest));
  ULA_CUDA(cudaStreamCreateWithPriority(&c->crit, cudaStreamNonBlocking, prio_greatest));
  ULA_CUDA(cudaStreamCreateWithPriority(&c->copy, cudaStreamNonBlocking, prio_greatest));
  ULA_CUDA(cudaStreamCreateWithPriority(&c->side, cudaStreamNonBlocking, prio_least));
  ULA_CUDA(cudaEventCreateWithFlags(&c->in_evt, cudaEventDisableTiming));
  uint32_t lmax = 0;
  for (uint32_t g = 0; g < G; ++g) lmax = cfg.layers_per_group[g] > lmax ? cfg.layers_per_group[g] : lmax;
  ULA_CUDA(resident_blocks(&c->move_blocks, &c->gather_blocks, lmax * cfg.row_bytes));
  c->gather_fit_per_sm = c->gather_blocks;
  // ULA_MOVE_BLOCKS_PER_SM / ULA_GATHER_BLOCKS_PER_SM tune the persistent grids
  // (clamped to what fits on an SM).
  c->move_blocks = env_blocks("ULA_MOVE_BLOCKS_PER_SM",
                              geo.cache ? ULA_CACHE_MOVE_BLOCKS : kMoveBlocksPerSm, c->move_blocks);
  c->gather_blocks = env_blocks("ULA_GATHER_BLOCKS_PER_SM", c->gather_blocks, c->gather_blocks);
  c->move_blocks *= c->sm_count;
  c->gather_blocks *= c->sm_count;
  c->emit_blocks = c->sm_count;
  c->stage_blocks = 2 * c->sm_count;

  // per-group step scratch and events
  const uint32_t max_blk = (cfg.max_entries + 255) / 256 + 1;
  c->steps.resize(G);
  for (uint32_t g = 0; g < G; ++g) {
    ula_ctx::GroupStep &st = c->steps[g];
    ULA_CUDA(c->alloc(&st.tbl, cfg.max_logical));
    ULA_CUDA(c->alloc(&st.addr_row, cfg.max_logical));
    ULA_CUDA(c->alloc(&st.blk, max_blk));
    ULA_CUDA(c->alloc(&st.miss_list, cfg.max_entries));
    ULA_CUDA(c->alloc(&st.miss_hs, cfg.max_entries));
    ULA_CUDA(c->alloc(&st.miss_row, cfg.max_entries));
    ULA_CUDA(c->alloc(&st.fill_order, c->decision_cap));
    ULA_CUDA(c->alloc(&st.vdone, c->decision_cap));
    ULA_CUDA(cudaMemsetAsync(st.vdone, 0, sizeof(uint32_t) * c->decision_cap, c->home));
    ULA_CUDA(cudaMemsetAsync(st.tbl, 0, sizeof(unsigned long long) * cfg.max_logical, c->home));
    for (cudaEvent_t *e : {&st.rot_evt, &st.meta_evt, &st.commit_evt, &st.hit_evt, &st.upd_evt})
      ULA_CUDA(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
    ULA_CUDA(cudaStreamCreateWithPriority(&st.upd, cudaStreamNonBlocking, prio_greatest));
  }
  ULA_CUDA(c->alloc(&c->status, 1));
  ULA_CUDA(c->alloc(&c->cnt_d, G));
  ULA_CUDA(c->alloc(&c->groups_d, G));
  if (H && !geo.cache && !geo.signal) {  // staged victim rows (the slot-major move only)
    const size_t rows = cfg.max_entries < S ? cfg.max_entries : S;  // victims per step <= both
    ULA_CUDA(c->alloc(&c->stage, rows * lmax * cfg.row_bytes));
  }
  ULA_CUDA(c->alloc(&c->spans_d, kSpanCap));
  cudaStream_t s = c->home;
  if (geo.exact) {  // one cooperative block per SM (it must fit beside the gathers)
    int per_sm = 0;
    ULA_CUDA(lru_resident_blocks(&per_sm));
    if (per_sm < 1) return ULA_ERR_CUDA;
    c->lru_blocks = c->sm_count;
    const size_t nb = (size_t)c->lru_blocks;
    ULA_CUDA(c->alloc(&c->lru.blk, 2 * nb));
    ULA_CUDA(c->alloc(&c->lru.hist, (size_t)kLruSelectPasses * kLruBins));
    ULA_CUDA(c->alloc(&c->lru.table, kSortBins * nb + kSortBins));
    ULA_CUDA(c->alloc(&c->lru.list[0], cfg.max_entries));
    ULA_CUDA(c->alloc(&c->lru.list[1], cfg.max_entries));
    ULA_CUDA(c->alloc(&c->lru.bar, 3));
    c->lru.per = (uint32_t)((((uint64_t)S + nb - 1) / nb + 3) & ~3ull);
    ULA_CUDA(c->alloc(&c->lru.rows, (size_t)kLruBins * nb));
    ULA_CUDA(c->alloc(&c->lru.totals, 2 * kLruBins));
    ULA_CUDA(cudaMemsetAsync(c->lru.totals, 0, 2 * kLruBins * sizeof(uint32_t), s));
    ULA_CUDA(c->alloc(&c->lru.blist, (size_t)c->lru.per * nb));
    ULA_CUDA(cudaMemsetAsync(c->lru.bar, 0, 3 * sizeof(uint32_t), s));
  }
  ULA_CUDA(cudaMemsetAsync(c->status, 0, sizeof(int), s));

  const uint32_t ncls = B + 2;
  const size_t work_len = (size_t)(B + 1) * geo.nseg + geo.hseg + 1;
  c->groups_h.resize(G);
  std::vector<GroupCounters> cnt_h(G);
  for (uint32_t g = 0; g < G; ++g) {
    GroupDev &d = c->groups_h[g];
    std::memset(&d, 0, sizeof(d));
    d.layers = cfg.layers_per_group[g];
    d.gpu_pool = gp[g];
    d.host_pool = H ? hp[g] : nullptr;
    ULA_CUDA(c->alloc(&d.map, cfg.max_logical));
    ULA_CUDA(c->alloc(&d.owner, S));
    ULA_CUDA(c->alloc(&d.stamp, S));
    ULA_CUDA(c->alloc(&d.cls0, (size_t)ncls * geo.gd.n0));
    ULA_CUDA(c->alloc(&d.cls1, (size_t)ncls * geo.gd.n1));
    ULA_CUDA(c->alloc(&d.cls2, (size_t)ncls * geo.gd.n2));
    ULA_CUDA(c->alloc(&d.clsc, (size_t)ncls * geo.gd.n1));
    ULA_CUDA(c->alloc(&d.hf0, geo.hd.n0));
    ULA_CUDA(c->alloc(&d.hf1, geo.hd.n1));
    ULA_CUDA(c->alloc(&d.hf2, geo.hd.n2));
    ULA_CUDA(c->alloc(&d.hfc, geo.hd.n1));
    ULA_CUDA(c->alloc(&d.uniq, cfg.max_entries));
    ULA_CUDA(c->alloc(&d.row_slot, cfg.max_entries));
    ULA_CUDA(c->alloc(&d.hitbits, geo.gd.n0));
    ULA_CUDA(cudaMemsetAsync(d.hitbits, 0, sizeof(uint32_t) * geo.gd.n0, s));
    ULA_CUDA(c->alloc(&d.victims, c->decision_cap));
    ULA_CUDA(c->alloc(&d.wb_host, c->decision_cap));
    ULA_CUDA(c->alloc(&d.work, work_len));
    d.cnt = c->cnt_d + g;
    if (geo.signal) {
      const uint32_t L = d.layers;
      ULA_CUDA(c->alloc(&d.layer_flag, L));
      ULA_CUDA(c->alloc(&d.layer_cnt, L));
      ULA_CUDA(c->alloc(&d.move_done, L + 1));  // [L]: the chunk dispenser
      ULA_CUDA(c->alloc(&d.gather_done, L));
      ULA_CUDA(c->alloc(&d.layer_ns, L + 1));
      ULA_CUDA(cudaMemsetAsync(d.layer_flag, 0, sizeof(uint32_t) * L, s));
      ULA_CUDA(cudaMemsetAsync(d.layer_cnt, 0, sizeof(uint32_t) * L, s));
      ULA_CUDA(cudaMemsetAsync(d.move_done, 0, sizeof(uint32_t) * (L + 1), s));
      ULA_CUDA(cudaMemsetAsync(d.gather_done, 0, sizeof(uint32_t) * L, s));
      ULA_CUDA(cudaMemsetAsync(d.layer_ns, 0, sizeof(unsigned long long) * (L + 1), s));
    }
    ULA_CUDA(cudaMemsetAsync(d.map, 0xff, sizeof(uint32_t) * cfg.max_logical, s));
    ULA_CUDA(cudaMemsetAsync(d.owner, 0xff, sizeof(uint32_t) * S, s));
    ULA_CUDA(cudaMemsetAsync(d.stamp, 0xff, sizeof(uint32_t) * S, s));
    ULA_CUDA(cudaMemsetAsync(d.cls0, 0, sizeof(uint32_t) * ncls * geo.gd.n0, s));
    ULA_CUDA(cudaMemsetAsync(d.cls1, 0, sizeof(uint32_t) * ncls * geo.gd.n1, s));
    ULA_CUDA(cudaMemsetAsync(d.cls2, 0, sizeof(uint32_t) * ncls * geo.gd.n2, s));
    ULA_CUDA(cudaMemsetAsync(d.clsc, 0, sizeof(uint32_t) * ncls * geo.gd.n1, s));
    ULA_CUDA(launch_bitmap_fill(class_bitmap(d, geo, B + 1), S, s));  // all slots free
    ULA_CUDA(launch_bitmap_fill(host_free_bitmap(d), H, s));
    std::memset(&cnt_h[g], 0, sizeof(GroupCounters));
    cnt_h[g].free_gpu = S;
    cnt_h[g].free_host = H;
  }
  ULA_CUDA(cudaMemcpyAsync(c->cnt_d, cnt_h.data(), sizeof(GroupCounters) * G,
                           cudaMemcpyHostToDevice, s));
  ULA_CUDA(cudaMemcpyAsync(c->groups_d, c->groups_h.data(), sizeof(GroupDev) * G,
                           cudaMemcpyHostToDevice, s));
  ULA_CUDA(cudaStreamSynchronize(s));
  c->live.assign(cfg.max_logical, 0);
  return ULA_OK;
}

}  // namespace

extern "C" {

const char *ula_error_string(int code) {
  switch (code) {
    case ULA_OK: return "ok";
    case ULA_ERR_INVALID_ARG: return "invalid argument";
    case ULA_ERR_CAPACITY: return "capacity exceeded";
    case ULA_ERR_UNMAPPED: return "selected address out of range or not allocated";
    case ULA_ERR_CUDA: return "CUDA runtime error";
    case ULA_ERR_TIMEOUT: return "bounded device wait expired";
    case ULA_ERR_POISONED: return "context poisoned by an earlier device-side error";
    case ULA_ERR_INTERNAL: return "device-side consistency check failed";
    default: return "unknown error";
  }
}

// internal_flags: kFlagCacheInternal for a TP rank's local buffer
static int create_ctx(const ula_config *cfg, void *const *gpu_pools, void *const *host_pools,
                      void *stream, uint32_t internal_flags, ula_ctx **out) {
  if (!out) return ULA_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc) return rc;
  ula_ctx *c = new ula_ctx;
  c->cfg = *cfg;
  c->cfg.flags |= internal_flags;
  c->home = static_cast<cudaStream_t>(stream);
  rc = create_impl(c, gpu_pools, host_pools);
  if (rc) {
    cudaDeviceSynchronize();
    destroy_resources(c);
    delete c;
    return rc;
  }
  *out = c;
  return ULA_OK;
}

int ula_create(const ula_config *cfg, void *const *gpu_pools, void *const *host_pools,
               void *stream, ula_ctx **out) {
  return create_ctx(cfg, gpu_pools, host_pools, stream, 0, out);
}

// rows: per group, `total` rows [total][L_g][W]; address i of this call is row
// phase + i * stride (stride 1, phase 0 for ula_alloc; a TP partition takes every
// P-th row of the TP call's range).
static int alloc_impl(ula_ctx *c, uint32_t n, const void *rows, uint32_t *logical_base,
                      uint32_t total, uint32_t phase, uint32_t stride) {
  if (!c || !logical_base) return ULA_ERR_INVALID_ARG;
  if (c->poisoned) return ULA_ERR_POISONED;
  const ula_config &cfg = c->cfg;
  if ((uint64_t)c->next_logical + n > cfg.max_logical) return ULA_ERR_CAPACITY;
  if (c->live_count + n > (uint64_t)cfg.gpu_slots + cfg.host_slots) return ULA_ERR_CAPACITY;
  *logical_base = c->next_logical;
  if (n == 0) return ULA_OK;
  ULA_CUDA(c->ensure_device());
  const uint8_t *rows_d =
      static_cast<const uint8_t *>(device_address(rows, c->device, true, true));
  if (!rows_d || !aligned16(rows_d)) return ULA_ERR_INVALID_ARG;
  // per group, on the group's update stream: after the group's last step only
  ULA_CUDA(cudaEventRecord(c->in_evt, c->home));
  const uint32_t base = c->next_logical;
  for (uint32_t g = 0; g < cfg.n_groups; ++g) {
    ULA_CUDA(c->begin_update(g));
    cudaStream_t s = c->steps[g].upd;
    unsigned long long acc = 0;  // byte offset of group g's rows
    for (uint32_t h = 0; h < g; ++h)
      acc += (unsigned long long)total * cfg.layers_per_group[h] * cfg.row_bytes;
    const unsigned long long sb = (unsigned long long)cfg.layers_per_group[g] * cfg.row_bytes;
    for (uint32_t off = 0; off < n; off += kAllocChunk) {
      const uint32_t m = n - off < kAllocChunk ? n - off : kAllocChunk;
      EmitParams sp{};
      sp.geo = c->geo;
      sp.groups = c->groups_d;
      sp.group0 = g;
      sp.order.n_cls = 1;
      sp.order.cls[0] = c->geo.B + 1;  // free slots only: alloc never evicts
      sp.quota = m;
      sp.status = c->status;
      ULA_CUDA(c->phase(ULA_PHASE_SELECT, s, 2, [&] {
        cudaError_t e = launch_alloc_select(sp, 1, s);
        return e != cudaSuccess ? e : launch_select_emit(sp, 1, c->emit_blocks, s);
      }));
      AllocParams ap{};
      ap.geo = c->geo;
      ap.groups = c->groups_d;
      ap.rows = rows_d;
      ap.group_off[g] = acc + ((unsigned long long)phase + (unsigned long long)off * stride) * sb;
      ap.round[g] = c->round[g];
      ap.group0 = g;
      ap.row_stride = stride;
      ap.base = base + off;
      ap.n = m;
      ap.status = c->status;
      ULA_CUDA(c->phase(ULA_PHASE_ALLOC, s, 1,
                        [&] { return launch_alloc_place(ap, 1, c->move_blocks, s); }));
    }
  }
  ULA_CUDA(c->end_updates(c->home));
  for (uint32_t i = 0; i < n; ++i) c->live[base + i] = 1;
  c->live_count += n;
  c->next_logical = base + n;
  return ULA_OK;
}

int ula_alloc(ula_ctx *c, uint32_t n, const void *rows, uint32_t *logical_base) {
  return alloc_impl(c, n, rows, logical_base, n, 0, 1);
}

// drop: a TP local buffer forgets any copies of [base, base + n) (no live check)
static int free_impl(ula_ctx *c, uint32_t base, uint32_t n, bool drop) {
  if (!c) return ULA_ERR_INVALID_ARG;
  if (c->poisoned) return ULA_ERR_POISONED;
  if (!drop) {
    if ((uint64_t)base + n > c->next_logical) return ULA_ERR_INVALID_ARG;
    for (uint32_t i = 0; i < n; ++i)
      if (!c->live[base + i]) return ULA_ERR_INVALID_ARG;
  } else if ((uint64_t)base + n > c->cfg.max_logical) {
    return ULA_ERR_INVALID_ARG;
  }
  if (n == 0) return ULA_OK;
  ULA_CUDA(c->ensure_device());
  ULA_CUDA(cudaEventRecord(c->in_evt, c->home));
  for (uint32_t g = 0; g < c->cfg.n_groups; ++g) {  // per group, after its last step only
    ULA_CUDA(c->begin_update(g));
    cudaStream_t s = c->steps[g].upd;
    FreeParams fp{};
    fp.geo = c->geo;
    fp.groups = c->groups_d;
    fp.round[g] = c->round[g];
    fp.group0 = g;
    fp.base = base;
    fp.n = n;
    fp.status = c->status;
    ULA_CUDA(c->phase(ULA_PHASE_FREE, s, 1, [&] { return launch_free(fp, 1, s); }));
  }
  ULA_CUDA(c->end_updates(c->home));
  if (!drop) {
    for (uint32_t i = 0; i < n; ++i) c->live[base + i] = 0;
    c->live_count -= n;
  }
  return ULA_OK;
}

int ula_free(ula_ctx *c, uint32_t base, uint32_t n) { return free_impl(c, base, n, false); }

int ula_step_group(ula_ctx *c, uint32_t group, const uint32_t *d_sel, uint32_t n_req, uint32_t q,
                   uint32_t k, void *d_out, uint32_t out_cap_rows, int32_t *d_entry_row,
                   int32_t *d_req_off, void *const *layer_ready, void *stream) {
  if (!c) return ULA_ERR_INVALID_ARG;
  if (c->poisoned) return ULA_ERR_POISONED;
  const ula_config &cfg = c->cfg;
  if (group >= cfg.n_groups) return ULA_ERR_INVALID_ARG;
  const uint64_t E = (uint64_t)n_req * q * k;
  if (E > cfg.max_entries) return ULA_ERR_INVALID_ARG;
  if (!d_req_off || (E && (!d_sel || !d_entry_row)) || (out_cap_rows && !d_out))
    return ULA_ERR_INVALID_ARG;
  if (d_out && !aligned16(d_out)) return ULA_ERR_INVALID_ARG;
  ULA_CUDA(c->ensure_device());
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  cudaStream_t s = c->crit;
  ula_ctx::GroupStep &st = c->steps[group];
  ULA_CUDA(c->enter(caller));
  if (st.in_flight) {  // this group's previous step: its move committed, its gather done
    ULA_CUDA(cudaStreamWaitEvent(s, st.commit_evt, 0));
    ULA_CUDA(cudaStreamWaitEvent(s, st.hit_evt, 0));
  }
  if (st.upd_pending) {  // and its last alloc/free
    ULA_CUDA(cudaStreamWaitEvent(s, st.upd_evt, 0));
    st.upd_pending = false;
  }

  if (++st.epoch == 0) {  // dedup stamps wrap: clear them
    ULA_CUDA(cudaMemsetAsync(st.tbl, 0, sizeof(unsigned long long) * cfg.max_logical, s));
    st.epoch = 1;
  }
  const uint32_t r = ++c->round[group];
  const uint32_t B = c->geo.B, cur = r % B;
  const GroupDev &gd = c->groups_h[group];

  StepParams p{};
  p.geo = c->geo;
  p.grp = gd;
  p.sel = d_sel;
  p.E = (uint32_t)E;
  p.QK = q * k;
  p.n_req = n_req;
  p.epoch = st.epoch;
  p.round = r;
  p.cur = cur;
  p.out_cap = out_cap_rows;
  const bool stall = c->inject == ULA_DEBUG_STALL_SCAN_BARRIER;
  p.inject = stall ? 0 : c->inject;
  p.entry_row = d_entry_row;
  p.req_off = d_req_off;
  p.tbl = st.tbl;
  p.addr_row = st.addr_row;
  p.blk = st.blk;
  p.miss_list = st.miss_list;
  p.miss_hs = st.miss_hs;
  p.miss_row = st.miss_row;
  p.src = c->tp_src[group];
  p.status = c->status;
  c->inject = 0;
  p.order.n_cls = B + 1;  // victims: free, cold, ring oldest (cur+1) .. newest (cur-1)
  p.order.cls[0] = B + 1;
  p.order.cls[1] = B;
  for (uint32_t d = 1; d < B; ++d) p.order.cls[1 + d] = (cur + d) % B;
  if (c->geo.exact) p.order.n_cls = 1;  // exact LRU walks the free slots; the scan does the rest
  SpanRec *meta_span = c->take_span(ULA_PHASE_SELECT, group);  // dedup .. victim emission
  p.span = meta_span;
  const bool gather = out_cap_rows != 0;
  GatherParams gp{};
  gp.geo = c->geo;
  gp.grp = gd;
  gp.out = static_cast<uint8_t *>(d_out);
  gp.out_cap = out_cap_rows;
  gp.layer = 0;
  gp.nlayers = gd.layers;
  gp.signal = c->geo.signal;
  gp.round = r;
  gp.status = c->status;
  // (6) the hit rows of every layer, one launch (a slot's layers are one contiguous
  // read); a hit's slot does not change in its round.  By default it is the first of
  // the step's copy kernels, so it never runs beside a move: the move's host-link
  // traffic holds up HBM traffic on every SM it shares (each slows the other).  With
  // ULA_FLAG_GATHER_BESIDE_MOVE (or the per-layer signal) it runs on the low-priority
  // side stream as soon as the compaction has recorded the hits' slots, beside the
  // marking, the victim selection and the move.
  auto launch_hit_gather = [&](cudaStream_t gs) -> cudaError_t {
    gp.span = c->take_span(ULA_PHASE_GATHER, group);
    return c->phase(ULA_PHASE_GATHER, gs, 1,
                    [&] { return launch_gather(gp, gather_step_blocks(E), gs); });
  };
  // (1)(2) dedup + translate + capacity check
  ULA_CUDA(c->phase(ULA_PHASE_DEDUP, s, E ? 2 : 1, [&] { return launch_dedup(p, s); }));
  // (3a) rotation + compaction of unique rows and misses
  ULA_CUDA(c->phase(ULA_PHASE_ROTATE, s, 1, [&] { return launch_rotate_emit(p, s); }));
  if (gather && c->beside) {
    ULA_CUDA(cudaEventRecord(st.rot_evt, s));
    ULA_CUDA(cudaStreamWaitEvent(c->side, st.rot_evt, 0));
    ULA_CUDA(launch_hit_gather(c->side));
    ULA_CUDA(cudaEventRecord(st.hit_evt, c->side));
  }
  // (3b) hits into the current bucket, entry rows; the victim walk
  ULA_CUDA(c->phase(ULA_PHASE_MARK, s, 1, [&] { return launch_mark_select(p, s); }));
  if (c->geo.exact) {
    // (4) exact LRU: the timestamp scan (a cooperative launch; its blocks fit on the
    // SMs beside the move's)
    LruParams lp{};
    lp.geo = c->geo;
    lp.grp = gd;
    lp.sc = c->lru;
    lp.round = r;
    lp.stall = stall ? 1 : 0;
    lp.status = c->status;
    ULA_CUDA(c->phase(ULA_PHASE_SELECT, s, 1,
                      [&] { return launch_lru_select(lp, c->lru_blocks, s); }));
  }
  // (4) victims' and write-back slots' indices; (5) the fill order
  const bool staged = !c->geo.signal;  // the slot-major move (not the layer-major one)
  EmitParams ep{};
  ep.geo = c->geo;
  ep.groups = c->groups_d;
  ep.group0 = group;
  ep.order = p.order;
  ep.quota = 0xffffffffu;
  ep.miss_hs = st.miss_hs;
  ep.fill_order = c->geo.signal ? nullptr : st.fill_order;
  ep.span = meta_span;
  ep.status = c->status;
  ULA_CUDA(c->phase(ULA_PHASE_SELECT, s, 1,
                    [&] { return launch_select_emit(ep, 1, c->emit_blocks, s); }));
  // the copies, on the copy stream after this step's metadata and after every earlier
  // call's copies
  cudaStream_t cs = c->copy;
  ULA_CUDA(cudaEventRecord(st.meta_evt, s));
  ULA_CUDA(cudaStreamWaitEvent(cs, st.meta_evt, 0));
  if (gather && !c->beside) ULA_CUDA(launch_hit_gather(cs));  // (its event after the move)
  // (5) write-back, fill (writing the missed rows' outputs), then map commit
  MoveParams mp{};
  mp.geo = c->geo;
  mp.grp = gd;
  mp.sel = d_sel;
  mp.entry_row = d_entry_row;
  mp.addr_row = st.addr_row;
  mp.E = (uint32_t)E;
  mp.miss_list = st.miss_list;
  mp.miss_hs = st.miss_hs;
  mp.miss_row = st.miss_row;
  mp.out = gather ? static_cast<uint8_t *>(d_out) : nullptr;
  mp.out_cap = out_cap_rows;
  mp.round = r;
  mp.cur = cur;
  mp.src = c->tp_src[group];
  mp.fill_order = st.fill_order;
  mp.stage = c->stage;
  mp.vdone = st.vdone;
  mp.status = c->status;
  if (staged) {  // entry rows; the rows of the victims that hold data, to the staging area
    mp.span = c->take_span(ULA_PHASE_STAGE, group);
    ULA_CUDA(c->phase(ULA_PHASE_STAGE, cs, 1, [&] { return launch_stage(mp, c->stage_blocks, cs); }));
  }
  mp.span = c->take_span(ULA_PHASE_MOVE, group);
  ULA_CUDA(c->phase(ULA_PHASE_MOVE, cs, c->geo.signal ? 2 : 1,
                    [&] { return launch_move(mp, c->move_blocks, staged, cs); }));
  // signal: the commit (and the hit gather) complete every layer of the output
  ULA_CUDA(cudaEventRecord(st.commit_evt, cs));
  // The gather's event: here when it ran on this stream (nothing stands between the
  // gather and the chained staging copy), or when there was nothing to gather.
  if (!gather || !c->beside) ULA_CUDA(cudaEventRecord(st.hit_evt, cs));
  st.in_flight = true;
  ULA_CUDA(cudaStreamWaitEvent(caller, st.commit_evt, 0));
  ULA_CUDA(cudaStreamWaitEvent(caller, st.hit_evt, 0));
  for (uint32_t j = 0; j < gd.layers; ++j)
    if (layer_ready && layer_ready[j])
      ULA_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(layer_ready[j]), caller));
  return ULA_OK;
}

static int sync_impl(ula_ctx *c) {
  ULA_CUDA(c->ensure_device());
  ULA_CUDA(cudaStreamSynchronize(c->crit));
  ULA_CUDA(cudaStreamSynchronize(c->copy));
  ULA_CUDA(cudaStreamSynchronize(c->side));
  for (auto &st : c->steps) ULA_CUDA(cudaStreamSynchronize(st.upd));
  ULA_CUDA(cudaStreamSynchronize(c->home));
  return ULA_OK;
}

int ula_sync(ula_ctx *c, ula_stats *stats) {
  if (!c) return ULA_ERR_INVALID_ARG;
  if (c->poisoned) return ULA_ERR_POISONED;
  int rc = sync_impl(c);
  if (rc) return rc;
  int st = 0;
  ULA_CUDA(cudaMemcpy(&st, c->status, sizeof(int), cudaMemcpyDeviceToHost));
  if (stats) {
    std::vector<GroupCounters> h(c->cfg.n_groups);
    ULA_CUDA(cudaMemcpy(h.data(), c->cnt_d, sizeof(GroupCounters) * h.size(),
                        cudaMemcpyDeviceToHost));
    unsigned long long acc[kStCount] = {};
    for (const GroupCounters &x : h)
      for (int i = 0; i < kStCount; ++i) acc[i] += x.stat[i];
    stats->steps = acc[kStSteps];
    stats->entries = acc[kStEntries];
    stats->uniq = acc[kStUniq];
    stats->hits = acc[kStHits];
    stats->misses = acc[kStMisses];
    stats->victims_free = acc[kStVictFree];
    stats->victims_cold = acc[kStVictCold];
    stats->victims_ring = acc[kStVictRing];
    stats->writebacks = acc[kStWriteback];
    stats->rows_gathered = acc[kStRows];
    stats->bytes_h2d = acc[kStBytesH2D];
    stats->bytes_d2h = acc[kStBytesD2H];
    stats->bypassed = acc[kStBypassed];
  }
  if (st) {
    c->poisoned = st;
    return st;
  }
  return ULA_OK;
}

void ula_destroy(ula_ctx *c) {
  if (!c) return;
  c->ensure_device();
  sync_impl(c);
  destroy_resources(c);
  delete c;
}

int ula_debug_layout_get(const ula_ctx *c, ula_debug_layout *out) {
  if (!c || !out) return ULA_ERR_INVALID_ARG;
  out->n0 = c->geo.gd.n0;
  out->n1 = c->geo.gd.n1;
  out->n2 = c->geo.gd.n2;
  out->h0 = c->geo.hd.n0;
  out->h1 = c->geo.hd.n1;
  out->h2 = c->geo.hd.n2;
  out->n_classes = c->geo.B + 2;
  out->decision_cap = c->decision_cap;
  return ULA_OK;
}

int ula_debug_export(ula_ctx *c, uint32_t group, ula_debug_state *st) {
  if (!c || !st || group >= c->cfg.n_groups) return ULA_ERR_INVALID_ARG;
  int rc = sync_impl(c);
  if (rc) return rc;
  const GroupDev &d = c->groups_h[group];
  const Geometry &geo = c->geo;
  const uint32_t ncls = geo.B + 2;
  auto copy = [&](void *dst, const void *src, size_t bytes) -> cudaError_t {
    if (!dst || !bytes) return cudaSuccess;
    return cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost);
  };
  ULA_CUDA(copy(st->map, d.map, sizeof(uint32_t) * c->cfg.max_logical));
  ULA_CUDA(copy(st->owner, d.owner, sizeof(uint32_t) * geo.S));
  ULA_CUDA(copy(st->stamp, d.stamp, sizeof(uint32_t) * geo.S));
  ULA_CUDA(copy(st->class_bits, d.cls0, sizeof(uint32_t) * ncls * geo.gd.n0));
  ULA_CUDA(copy(st->class_sum1, d.cls1, sizeof(uint32_t) * ncls * geo.gd.n1));
  ULA_CUDA(copy(st->class_sum2, d.cls2, sizeof(uint32_t) * ncls * geo.gd.n2));
  ULA_CUDA(copy(st->host_free_bits, d.hf0, sizeof(uint32_t) * geo.hd.n0));
  ULA_CUDA(copy(st->host_free_sum1, d.hf1, sizeof(uint32_t) * geo.hd.n1));
  ULA_CUDA(copy(st->host_free_sum2, d.hf2, sizeof(uint32_t) * geo.hd.n2));
  ULA_CUDA(copy(st->class_seg_count, d.clsc, sizeof(uint32_t) * ncls * geo.gd.n1));
  ULA_CUDA(copy(st->host_seg_count, d.hfc, sizeof(uint32_t) * geo.hd.n1));
  ULA_CUDA(copy(st->row_slot, d.row_slot, sizeof(uint32_t) * c->cfg.max_entries));
  ULA_CUDA(copy(st->uniq, d.uniq, sizeof(uint32_t) * c->cfg.max_entries));
  ULA_CUDA(copy(st->victims, d.victims, sizeof(uint32_t) * c->decision_cap));
  ULA_CUDA(copy(st->wb_host, d.wb_host, sizeof(uint32_t) * c->decision_cap));
  GroupCounters cnt;
  ULA_CUDA(cudaMemcpy(&cnt, d.cnt, sizeof(cnt), cudaMemcpyDeviceToHost));
  st->round = c->round[group];
  st->cur = c->round[group] % geo.B;
  st->free_gpu = cnt.free_gpu;
  st->free_host = cnt.free_host;
  st->U = cnt.U;
  st->M = cnt.M;
  st->hits = cnt.hits;
  st->victims_free = cnt.F;
  st->writebacks = cnt.K;
  return ULA_OK;
}

int ula_profile_enable(ula_ctx *c, int on) {
  if (!c) return ULA_ERR_INVALID_ARG;
  c->prof_on = on != 0;
  return ULA_OK;
}

int ula_profile_read(ula_ctx *c, ula_profile *out, int reset) {
  if (!c) return ULA_ERR_INVALID_ARG;
  int rc = sync_impl(c);
  if (rc) return rc;
  for (auto &t : c->prof_pending) {
    float ms = 0.f;
    ULA_CUDA(cudaEventElapsedTime(&ms, t.a, t.b));
    c->prof_ms[t.phase] += ms;
    c->prof_timed[t.phase] += 1;
    c->prof_spare.push_back(t.a);
    c->prof_spare.push_back(t.b);
  }
  c->prof_pending.clear();
  if (out) {
    for (int i = 0; i < ULA_PHASE_COUNT; ++i) {
      out->kernels[i] = c->prof_kernels[i];
      out->timed[i] = c->prof_timed[i];
      out->ms[i] = c->prof_ms[i];
    }
  }
  if (reset) {
    for (int i = 0; i < ULA_PHASE_COUNT; ++i) {
      c->prof_kernels[i] = 0;
      c->prof_timed[i] = 0;
      c->prof_ms[i] = 0.0;
    }
  }
  return ULA_OK;
}

static cudaError_t reset_spans(ula_ctx *c) {
  c->span_meta.clear();
  return cudaMemset(c->spans_d, 0xff, sizeof(SpanRec) * kSpanCap);
}

int ula_profile_spans(ula_ctx *c, int on) {
  if (!c) return ULA_ERR_INVALID_ARG;
  int rc = sync_impl(c);
  if (rc) return rc;
  ULA_CUDA(reset_spans(c));
  c->span_on = on != 0;
  return ULA_OK;
}

int ula_profile_spans_read(ula_ctx *c, ula_span *out, uint32_t cap, uint32_t *count) {
  if (!c || !count || (cap && !out)) return ULA_ERR_INVALID_ARG;
  int rc = sync_impl(c);
  if (rc) return rc;
  const size_t n = c->span_meta.size();
  *count = (uint32_t)n;
  const size_t k = n < cap ? n : cap;
  if (k) {
    std::vector<SpanRec> h(k);
    ULA_CUDA(cudaMemcpy(h.data(), c->spans_d, sizeof(SpanRec) * k, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < k; ++i) {
      out[i].phase = c->span_meta[i] >> 16;
      out[i].group = c->span_meta[i] & 0xffffu;
      const bool ran = h[i].t0 != ~0ull && h[i].t1n != ~0ull;
      out[i].start_ns = ran ? h[i].t0 : 0;
      out[i].end_ns = ran ? ~h[i].t1n : 0;
    }
  }
  ULA_CUDA(reset_spans(c));
  return ULA_OK;
}

int ula_debug_regather(ula_ctx *c, uint32_t group, uint32_t layer, uint32_t n_layers,
                       void *d_out, uint32_t out_cap_rows, uint32_t blocks_per_sm, void *stream) {
  if (!c || group >= c->cfg.n_groups || !d_out || !aligned16(d_out)) return ULA_ERR_INVALID_ARG;
  if (c->poisoned) return ULA_ERR_POISONED;
  const GroupDev &gd = c->groups_h[group];
  if (layer >= gd.layers || n_layers < 1 || n_layers > gd.layers - layer || out_cap_rows < 1)
    return ULA_ERR_INVALID_ARG;
  ULA_CUDA(c->ensure_device());
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  GatherParams gp{};
  gp.geo = c->geo;
  gp.grp = gd;
  gp.out = static_cast<uint8_t *>(d_out);
  gp.out_cap = out_cap_rows;
  gp.layer = layer;
  gp.nlayers = n_layers;
  gp.status = c->status;
  int blocks = gather_step_blocks(c->cfg.max_entries);
  if (blocks_per_sm) {
    const int fit = c->gather_fit_per_sm;
    blocks = c->sm_count * ((int)blocks_per_sm < fit ? (int)blocks_per_sm : fit);
  }
  ULA_CUDA(launch_gather(gp, blocks, caller));
  return ULA_OK;
}

int ula_layer_signal(ula_ctx *c, uint32_t group, const uint32_t **d_flags, uint32_t *round) {
  if (!c || !d_flags || !round || !c->geo.signal || group >= c->cfg.n_groups)
    return ULA_ERR_INVALID_ARG;
  *d_flags = c->groups_h[group].layer_flag;
  *round = c->round[group];
  return ULA_OK;
}

int ula_debug_layer_times(ula_ctx *c, uint32_t group, unsigned long long *ns) {
  if (!c || !ns || !c->geo.signal || group >= c->cfg.n_groups) return ULA_ERR_INVALID_ARG;
  if (c->poisoned) return ULA_ERR_POISONED;
  int rc = sync_impl(c);
  if (rc) return rc;
  const GroupDev &d = c->groups_h[group];
  ULA_CUDA(cudaMemcpy(ns, d.layer_ns, sizeof(unsigned long long) * (d.layers + 1),
                      cudaMemcpyDeviceToHost));
  return ULA_OK;
}

int ula_debug_consume(ula_ctx *c, uint32_t group, uint32_t layer, uint32_t round,
                      const void *d_out, uint32_t out_cap_rows, uint32_t n_rows,
                      unsigned long long *d_result, void *stream) {
  if (!c || !c->geo.signal || group >= c->cfg.n_groups || !d_result) return ULA_ERR_INVALID_ARG;
  const GroupDev &d = c->groups_h[group];
  if (layer >= d.layers || n_rows > out_cap_rows || (n_rows && !d_out)) return ULA_ERR_INVALID_ARG;
  if (c->poisoned) return ULA_ERR_POISONED;
  ULA_CUDA(c->ensure_device());
  ULA_CUDA(launch_consume(d.layer_flag + layer, round, static_cast<const uint8_t *>(d_out),
                          out_cap_rows, layer, n_rows, c->cfg.row_bytes, d_result,
                          static_cast<cudaStream_t>(stream)));
  return ULA_OK;
}

int ula_debug_inject(ula_ctx *c, int code) {
  if (!c) return ULA_ERR_INVALID_ARG;
  if (c->poisoned) return ULA_ERR_POISONED;
  c->inject = code;
  return ULA_OK;
}


// ------------------------------------------------------------------ TP mode

struct ula_tp {
  uint32_t P = 0, G = 0;
  ula_config cfg{};
  std::vector<ula_ctx *> parts, bufs;
  std::vector<cudaStream_t> ps, bs;
  std::vector<cudaEvent_t> pdone, bdone;
  cudaEvent_t split_evt = nullptr;
  uint32_t *sel = nullptr;  // [2P][max_entries]: partitions' entries, then buffers'
  uint32_t next_logical = 0;
};

static void tp_release(ula_tp *t) {
  for (ula_ctx *c : t->parts) ula_destroy(c);
  for (ula_ctx *c : t->bufs) ula_destroy(c);
  for (cudaStream_t s : t->ps) cudaStreamDestroy(s);
  for (cudaStream_t s : t->bs) cudaStreamDestroy(s);
  for (cudaEvent_t e : t->pdone) cudaEventDestroy(e);
  for (cudaEvent_t e : t->bdone) cudaEventDestroy(e);
  if (t->split_evt) cudaEventDestroy(t->split_evt);
  if (t->sel) cudaFree(t->sel);
  delete t;
}

int ula_tp_create(const ula_config *cfg, uint32_t parts, uint32_t buffer_slots,
                  void *const *gpu_pools, void *const *host_pools, void *const *buffer_pools,
                  void *stream, ula_tp **out) {
  if (!out || !cfg || parts == 0 || parts > kMaxParts || buffer_slots == 0 || !gpu_pools ||
      !buffer_pools)
    return ULA_ERR_INVALID_ARG;
  *out = nullptr;
  if (cfg->flags & (ULA_FLAG_LAYER_SIGNAL | ULA_FLAG_EXACT_LRU)) return ULA_ERR_INVALID_ARG;
  int rc = validate_config(cfg);
  if (rc) return rc;
  ula_tp *t = new ula_tp;
  t->P = parts;
  t->G = cfg->n_groups;
  t->cfg = *cfg;
  const uint32_t G = t->G;
  ula_config pc = *cfg;  // a partition: local ids
  pc.max_logical = (cfg->max_logical + parts - 1) / parts;
  ula_config bc = *cfg;  // a buffer: global addresses, no host pool
  bc.gpu_slots = buffer_slots;
  bc.host_slots = 0;
  bc.flags = 0;
  for (uint32_t p = 0; p < parts && !rc; ++p) {
    ula_ctx *c = nullptr;
    rc = create_ctx(&pc, gpu_pools + (size_t)p * G, host_pools ? host_pools + (size_t)p * G : nullptr,
                    stream, 0, &c);
    if (!rc) t->parts.push_back(c);
  }
  for (uint32_t r = 0; r < parts && !rc; ++r) {
    ula_ctx *c = nullptr;
    rc = create_ctx(&bc, buffer_pools + (size_t)r * G, nullptr, stream, kFlagCacheInternal, &c);
    if (!rc) t->bufs.push_back(c);
  }
  cudaError_t e = cudaSuccess;
  for (uint32_t p = 0; p < parts && !rc && e == cudaSuccess; ++p) {
    cudaStream_t a = nullptr, b = nullptr;
    cudaEvent_t x = nullptr, y = nullptr;
    e = cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking);
    if (e == cudaSuccess) t->ps.push_back(a), e = cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking);
    if (e == cudaSuccess) t->bs.push_back(b), e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
    if (e == cudaSuccess) t->pdone.push_back(x), e = cudaEventCreateWithFlags(&y, cudaEventDisableTiming);
    if (e == cudaSuccess) t->bdone.push_back(y);
  }
  if (!rc && e == cudaSuccess) e = cudaEventCreateWithFlags(&t->split_evt, cudaEventDisableTiming);
  if (!rc && e == cudaSuccess)
    e = cudaMalloc(&t->sel, sizeof(uint32_t) * 2 * (size_t)parts * cfg->max_entries);
  if (!rc && e != cudaSuccess) rc = ULA_ERR_CUDA;
  if (!rc) {  // every buffer fetches from the partitions' maps and GPU pools
    for (ula_ctx *b : t->bufs)
      for (uint32_t g = 0; g < G; ++g) {
        TpSource &src = b->tp_src[g];
        src.P = parts;
        src.S = cfg->gpu_slots;
        for (uint32_t p = 0; p < parts; ++p) {
          src.map[p] = t->parts[p]->groups_h[g].map;
          src.pool[p] = t->parts[p]->groups_h[g].gpu_pool;
        }
      }
  }
  if (rc) {
    cudaDeviceSynchronize();
    tp_release(t);
    return rc;
  }
  *out = t;
  return ULA_OK;
}

int ula_tp_alloc(ula_tp *t, uint32_t n, const void *rows, uint32_t *logical_base) {
  if (!t || !logical_base) return ULA_ERR_INVALID_ARG;
  if ((uint64_t)t->next_logical + n > t->cfg.max_logical) return ULA_ERR_CAPACITY;
  const uint32_t base = t->next_logical;
  for (uint32_t p = 0; p < t->P; ++p) {
    uint32_t first = base;
    while (first < base + n && first % t->P != p) ++first;
    const uint32_t cnt = first < base + n ? (base + n - first + t->P - 1) / t->P : 0;
    uint32_t lb = 0;
    const int rc = alloc_impl(t->parts[p], cnt, rows, &lb, n, first - base, t->P);
    if (rc) return rc;
    if (cnt && lb != first / t->P) return ULA_ERR_INTERNAL;
  }
  t->next_logical = base + n;
  *logical_base = base;
  return ULA_OK;
}

int ula_tp_free(ula_tp *t, uint32_t base, uint32_t n) {
  if (!t || (uint64_t)base + n > t->next_logical) return ULA_ERR_INVALID_ARG;
  for (uint32_t p = 0; p < t->P; ++p) {
    uint32_t first = base;
    while (first < base + n && first % t->P != p) ++first;
    const uint32_t cnt = first < base + n ? (base + n - first + t->P - 1) / t->P : 0;
    if (cnt) {
      const int rc = free_impl(t->parts[p], first / t->P, cnt, false);
      if (rc) return rc;
    }
  }
  for (ula_ctx *b : t->bufs) {
    const int rc = free_impl(b, base, n, true);
    if (rc) return rc;
  }
  return ULA_OK;
}

int ula_tp_step_group(ula_tp *t, uint32_t group, const uint32_t *d_sel, uint32_t n_req,
                      uint32_t q, uint32_t k, void *const *d_local_out,
                      void *const *d_remote_out, uint32_t out_cap_rows,
                      int32_t *const *d_local_entry_row, int32_t *const *d_local_req_off,
                      int32_t *const *d_remote_entry_row, int32_t *const *d_remote_req_off,
                      void *stream) {
  if (!t || group >= t->G || !d_local_out || !d_remote_out || !d_local_entry_row ||
      !d_local_req_off || !d_remote_entry_row || !d_remote_req_off)
    return ULA_ERR_INVALID_ARG;
  const uint64_t E = (uint64_t)n_req * q * k;
  if (E > t->cfg.max_entries || (E && !d_sel)) return ULA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint32_t P = t->P, stride = t->cfg.max_entries;
  uint32_t *part_sel = t->sel, *buf_sel = t->sel + (size_t)P * stride;
  ula_ctx *c0 = t->parts[0];
  ula_ctx *c = c0;  // (for ULA_CUDA's error path)
  ULA_CUDA(launch_tp_split(d_sel, (uint32_t)E, P, part_sel, buf_sel, stride, s));
  ULA_CUDA(cudaEventRecord(t->split_evt, s));
  for (uint32_t p = 0; p < P; ++p) {  // the partitions, concurrently
    c = t->parts[p];
    ULA_CUDA(cudaStreamWaitEvent(t->ps[p], t->split_evt, 0));
    const int rc = ula_step_group(c, group, part_sel + (size_t)p * stride, n_req, q, k,
                                  d_local_out[p], out_cap_rows, d_local_entry_row[p],
                                  d_local_req_off[p], nullptr, t->ps[p]);
    if (rc) return rc;
    ULA_CUDA(cudaEventRecord(t->pdone[p], t->ps[p]));
  }
  for (uint32_t r = 0; r < P; ++r) {  // then every rank's buffer fetches from them
    c = t->bufs[r];
    for (uint32_t p = 0; p < P; ++p) ULA_CUDA(cudaStreamWaitEvent(t->bs[r], t->pdone[p], 0));
    const int rc = ula_step_group(c, group, buf_sel + (size_t)r * stride, n_req, q, k,
                                  d_remote_out[r], out_cap_rows, d_remote_entry_row[r],
                                  d_remote_req_off[r], nullptr, t->bs[r]);
    if (rc) return rc;
    ULA_CUDA(cudaEventRecord(t->bdone[r], t->bs[r]));
  }
  c = c0;
  for (uint32_t r = 0; r < P; ++r) ULA_CUDA(cudaStreamWaitEvent(s, t->bdone[r], 0));
  return ULA_OK;
}

int ula_tp_sync(ula_tp *t, ula_stats *stats) {
  if (!t) return ULA_ERR_INVALID_ARG;
  int first = ULA_OK;
  for (uint32_t i = 0; i < 2 * t->P; ++i) {
    ula_ctx *c = i < t->P ? t->parts[i] : t->bufs[i - t->P];
    const int rc = ula_sync(c, stats ? stats + i : nullptr);
    if (rc && !first) first = rc;
  }
  return first;
}

ula_ctx *ula_tp_context(ula_tp *t, int kind, uint32_t index) {
  if (!t || index >= t->P || (kind != 0 && kind != 1)) return nullptr;
  return kind == 0 ? t->parts[index] : t->bufs[index];
}

int ula_tp_destroy(ula_tp *t) {
  if (!t) return ULA_ERR_INVALID_ARG;
  for (ula_ctx *c : t->parts) sync_impl(c);
  for (ula_ctx *c : t->bufs) sync_impl(c);
  tp_release(t);
  return ULA_OK;
}

}  // extern "C"
