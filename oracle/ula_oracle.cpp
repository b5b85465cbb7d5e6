// TEST INFRASTRUCTURE -- the CPU oracle of the KV residency path.
//
// Only the tests, the smoke check and the benchmark's CPU-baseline leg may
// load this library.  It shares no code with the CUDA path: it keeps its own
// containers (one ordered set per slot class, a per-address location record)
// and walks the method's steps one by one, in the order the pages give them.
// It is slow on purpose and single-threaded.
//
// Source: "UlaCache: Unified Logical Addressing for Sparse LLM Serving"
// (paper summary page).
//   §2 "Unified logical addresses": every KV entry has a fixed logical
//       address and a mapping entry naming the GPU slot or the CPU slot that
//       holds it; in DP mode an entry lives on the GPU or on the CPU, never
//       both; a layer group sharing one selection does lookup and dedup once.
//   §3 "PB-LRU": slots accessed in one scheduling round go into one bucket;
//       each layer group keeps a ring of buckets plus a cold bucket; each
//       round the current bucket advances one position and what is left in
//       the bucket about to be reused goes to the cold bucket (labels only);
//       space comes from free slots, then the cold bucket, then the ring from
//       oldest to newest; the current bucket is never chosen; data moves
//       first, then the mapping is updated, then completion is signalled.
//
// Readings where the pages are silent:
//   * one GPU slot holds the rows of all L_g layers of one address for one
//     group; each group has its own map, pools, ring and cold bucket;
//   * one scheduling round = one step call for that group; rotation happens
//     at the start of the round, before hits are marked;
//   * the ring has B buckets including the current one; the oldest ring
//     bucket is cur+1, the newest cur-1 (mod B);
//   * inside every class, the lowest slot index goes first;
//   * dedup keeps first occurrences in flattened (request, query, i) order;
//     the i-th miss in that order gets the i-th victim;
//   * the j-th victim that holds data is written back to the j-th lowest
//     host slot free before the step; the misses' host slots are released
//     after all moves;
//   * a step needing more victims than S - hits, more host slots than are
//     free, or more output rows than the caller's buffer fails with
//     CAPACITY before any state changes; an unallocated or out-of-range
//     address fails with UNMAPPED before any state changes;
//   * alloc hands out logical bases monotonically, places each new address
//     in the lowest free GPU slot (joining the current bucket), else the
//     lowest free host slot, and never evicts; free releases both tiers;
//   * with the overflow bypass enabled (an extension, not on the pages), a
//     step with more misses than can be made resident moves only the first
//     M' = min(M, S - hits, free GPU + free host slots) misses; each later
//     miss is gathered straight from its host slot into the output and stays
//     on the host;
//   * TP mode (emulated, orc_tp_*): address t belongs to partition t mod P, a
//     DP residency over local ids t / P; each rank keeps per group a local
//     buffer of remote rows (PB-LRU over its own slots and ring, victims'
//     copies dropped, misses fetched from the owner's GPU slot after the
//     owner's step);
//   * exact LRU (the baseline policy of §3's first paragraph, selectable in
//     place of PB-LRU): every GPU slot keeps a timestamp, the round of its
//     last access (a hit, a fill, or an alloc placement, which counts in the
//     latest round); victims are the free slots, lowest first, then the
//     occupied slots in ascending (timestamp, slot) order.  A slot accessed in
//     the current round is never chosen.  There are no buckets: every
//     occupied slot carries the one label "cold".  Everything else (pairing,
//     write-back slots, capacity, bypass, move -> map -> signal) is as above.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

namespace {

constexpr uint32_t kPad = 0xFFFFFFFFu;
constexpr uint32_t kNone = 0xFFFFFFFFu;

// Status values (same numbers as the library's documented error codes).
enum {
  kOk = 0,
  kInvalidArg = 1,
  kCapacity = 2,
  kUnmapped = 3,
  kInternal = 7,  // a guard that cannot fire when the steps above are right
};

// Slot class labels.
constexpr int kFree = -1;
constexpr int kCold = -2;

enum Tier : uint8_t { kUnallocated = 0, kOnGpu = 1, kOnHost = 2 };

struct Location {
  Tier tier = kUnallocated;
  uint32_t slot = 0;
};

struct Group {
  uint32_t layers = 0;
  std::vector<Location> where;          // [max_logical]: the logical-to-physical map
  std::vector<int> cls;                 // [S]: kFree, kCold or a ring bucket index
  std::vector<uint32_t> stamp;          // [S]: round of the last access, kNone if free
  std::set<std::pair<uint32_t, uint32_t>> by_age;  // exact LRU: (stamp, slot) of occupied slots
  uint32_t round = 0;                   // scheduling rounds (step calls) so far
  std::vector<uint32_t> owner;          // [S]: logical address held, or kNone
  std::set<uint32_t> free_slots;        // GPU slots holding nothing
  std::set<uint32_t> cold;              // the cold bucket
  std::vector<std::set<uint32_t>> ring; // [B] ring buckets
  uint32_t cur = 0;                     // current ring bucket
  std::set<uint32_t> host_free;         // free host slots
  std::vector<uint32_t> host_owner;     // [H]
  std::vector<uint8_t> gpu_pool;        // [S][layers][row_bytes]
  std::vector<uint8_t> host_pool;       // [H][layers][row_bytes]
  // decisions of the last step (for inspection by tests)
  std::vector<uint32_t> last_victims;   // victim i paired with miss i
  std::vector<uint32_t> last_wb_host;   // host slot of the j-th write-back
  std::vector<int> last_victim_class;   // class each victim was taken from
  size_t last_bypassed = 0;             // misses served from the host pool directly
};

constexpr uint32_t kFlagBypass = 1u;    // overflow bypass (same bits as the library's flags)
constexpr uint32_t kFlagExactLru = 2u;  // exact LRU in place of PB-LRU

struct Oracle {
  uint32_t row_bytes = 0, n_groups = 0, S = 0, H = 0, B = 0, max_logical = 0, flags = 0;
  uint32_t next_logical = 0;
  std::vector<uint8_t> live;  // [max_logical]
  std::vector<Group> groups;

  size_t slot_bytes(const Group &g) const { return (size_t)g.layers * row_bytes; }
  bool exact() const { return (flags & kFlagExactLru) != 0; }
};

void remove_from_class(Group &g, uint32_t s) {
  int c = g.cls[s];
  if (c == kFree) g.free_slots.erase(s);
  else if (c == kCold) g.cold.erase(s);
  else g.ring[(size_t)c].erase(s);
}

void move_to_current_bucket(Group &g, uint32_t s) {
  remove_from_class(g, s);
  g.ring[g.cur].insert(s);
  g.cls[s] = (int)g.cur;
}

// Slot s is accessed in the current round: PB-LRU moves it into the current
// bucket; exact LRU renews its timestamp (it joins, or stays in, the one
// occupied class).
void touch(const Oracle &o, Group &g, uint32_t s) {
  if (o.exact()) {
    if (g.cls[s] != kFree) g.by_age.erase({g.stamp[s], s});
    remove_from_class(g, s);
    g.cold.insert(s);
    g.cls[s] = kCold;
    g.by_age.insert({g.round, s});
  } else {
    move_to_current_bucket(g, s);
  }
  g.stamp[s] = g.round;
}

// Slot s gives up its data and becomes free.
void release_slot(Group &g, uint32_t s) {
  if (g.cls[s] != kFree) g.by_age.erase({g.stamp[s], s});
  remove_from_class(g, s);
  g.free_slots.insert(s);
  g.cls[s] = kFree;
  g.owner[s] = kNone;
  g.stamp[s] = kNone;
}

}  // namespace

extern "C" {

void *orc_create2(uint32_t row_bytes, uint32_t n_groups, const uint32_t *layers, uint32_t S,
                  uint32_t H, uint32_t B, uint32_t max_logical, uint32_t flags) {
  if (!row_bytes || !n_groups || !layers || !S || !B || !max_logical) return nullptr;
  if (flags & ~(kFlagBypass | kFlagExactLru)) return nullptr;
  Oracle *o = new Oracle;
  o->flags = flags;
  o->row_bytes = row_bytes;
  o->n_groups = n_groups;
  o->S = S;
  o->H = H;
  o->B = B;
  o->max_logical = max_logical;
  o->live.assign(max_logical, 0);
  o->groups.resize(n_groups);
  for (uint32_t gi = 0; gi < n_groups; ++gi) {
    Group &g = o->groups[gi];
    g.layers = layers[gi];
    g.where.assign(max_logical, Location{});
    g.cls.assign(S, kFree);
    g.stamp.assign(S, kNone);
    g.owner.assign(S, kNone);
    for (uint32_t s = 0; s < S; ++s) g.free_slots.insert(s);
    g.ring.assign(B, std::set<uint32_t>{});
    g.cur = 0;
    for (uint32_t h = 0; h < H; ++h) g.host_free.insert(h);
    g.host_owner.assign(H, kNone);
    g.gpu_pool.assign((size_t)S * o->slot_bytes(g), 0);
    g.host_pool.assign((size_t)H * o->slot_bytes(g), 0);
  }
  return o;
}

void *orc_create(uint32_t row_bytes, uint32_t n_groups, const uint32_t *layers, uint32_t S,
                 uint32_t H, uint32_t B, uint32_t max_logical) {
  return orc_create2(row_bytes, n_groups, layers, S, H, B, max_logical, 0);
}

void orc_destroy(void *h) { delete static_cast<Oracle *>(h); }

// rows: for each group in order, [n][layers_g][row_bytes] (groups concatenated).
int orc_alloc(void *h, uint32_t n, const uint8_t *rows, uint32_t *base_out) {
  Oracle *o = static_cast<Oracle *>(h);
  if (!o || !base_out || (n && !rows)) return kInvalidArg;
  if ((uint64_t)o->next_logical + n > o->max_logical) return kCapacity;
  for (const Group &g : o->groups)
    if ((size_t)n > g.free_slots.size() + g.host_free.size()) return kCapacity;
  const uint32_t base = o->next_logical;
  size_t group_off = 0;
  for (Group &g : o->groups) {
    const size_t sb = o->slot_bytes(g);
    for (uint32_t i = 0; i < n; ++i) {
      const uint32_t a = base + i;
      const uint8_t *src = rows + group_off + (size_t)i * sb;
      if (!g.free_slots.empty()) {  // lowest free GPU slot; a prefill write counts as an access
        uint32_t s = *g.free_slots.begin();
        touch(*o, g, s);
        g.owner[s] = a;
        g.where[a] = Location{kOnGpu, s};
        std::memcpy(&g.gpu_pool[(size_t)s * sb], src, sb);
      } else {  // otherwise the lowest free host slot
        uint32_t hs = *g.host_free.begin();
        g.host_free.erase(hs);
        g.host_owner[hs] = a;
        g.where[a] = Location{kOnHost, hs};
        std::memcpy(&g.host_pool[(size_t)hs * sb], src, sb);
      }
    }
    group_off += (size_t)n * sb;
  }
  for (uint32_t i = 0; i < n; ++i) o->live[base + i] = 1;
  o->next_logical = base + n;
  *base_out = base;
  return kOk;
}

int orc_free(void *h, uint32_t base, uint32_t n) {
  Oracle *o = static_cast<Oracle *>(h);
  if (!o || (uint64_t)base + n > o->max_logical) return kInvalidArg;
  for (uint32_t i = 0; i < n; ++i)
    if (!o->live[base + i]) return kInvalidArg;
  for (Group &g : o->groups) {
    for (uint32_t i = 0; i < n; ++i) {
      const uint32_t a = base + i;
      Location loc = g.where[a];
      if (loc.tier == kOnGpu) {
        release_slot(g, loc.slot);
      } else {
        g.host_free.insert(loc.slot);
        g.host_owner[loc.slot] = kNone;
      }
      g.where[a] = Location{};
    }
  }
  for (uint32_t i = 0; i < n; ++i) o->live[base + i] = 0;
  return kOk;
}

// counters (optional, [9]): uniq, hits, misses, victims from free, from cold,
// from the ring, write-backs, rows gathered, misses bypassed.
int orc_step_group(void *h, uint32_t gi, const uint32_t *sel, uint32_t n_req, uint32_t q,
                   uint32_t k, uint8_t *out, uint32_t out_cap, int32_t *entry_row,
                   int32_t *req_off, uint64_t *counters) {
  Oracle *o = static_cast<Oracle *>(h);
  if (!o || gi >= o->n_groups || (n_req && (!sel || !entry_row || !req_off))) return kInvalidArg;
  Group &g = o->groups[gi];
  const size_t E = (size_t)n_req * q * k;
  const size_t sb = o->slot_bytes(g);

  // (1) dedup: one lookup per distinct address of the group's shared selection,
  //     first occurrences kept in flattened (request, query, i) order.
  std::vector<uint32_t> uniq;
  std::unordered_map<uint32_t, int32_t> row_of;
  row_of.reserve(E * 2 + 1);
  for (uint32_t r = 0; r < n_req; ++r) {
    req_off[r] = (int32_t)uniq.size();
    for (size_t e = (size_t)r * q * k; e < (size_t)(r + 1) * q * k; ++e) {
      const uint32_t a = sel[e];
      if (a == kPad) continue;
      if (a >= o->max_logical || g.where[a].tier == kUnallocated) return kUnmapped;
      if (row_of.find(a) == row_of.end()) {
        row_of.emplace(a, (int32_t)uniq.size());
        uniq.push_back(a);
      }
    }
  }
  req_off[n_req] = (int32_t)uniq.size();

  // (2) translate through the map: GPU-resident = hit, host-resident = miss.
  std::vector<uint32_t> misses, bypassed;
  size_t hits = 0;
  for (uint32_t a : uniq) {
    if (g.where[a].tier == kOnGpu) ++hits;
    else misses.push_back(a);
  }
  // capacity: victims come from everything but the current bucket, which
  // after marking holds exactly the hits; write-backs need free host slots.
  const size_t free_gpu = g.free_slots.size();
  const size_t can_place = std::min((size_t)o->S - hits, free_gpu + g.host_free.size());
  if (uniq.size() > out_cap) return kCapacity;
  if (misses.size() > can_place) {
    if (!(o->flags & kFlagBypass)) return kCapacity;
    // bypass: only the first can_place misses become resident; the rest are
    // gathered from the host pool below and stay where they are
    bypassed.assign(misses.begin() + can_place, misses.end());
    misses.resize(can_place);
  }
  const size_t M = misses.size();
  const size_t writebacks_needed = M > free_gpu ? M - free_gpu : 0;

  for (size_t e = 0; e < E; ++e) entry_row[e] = sel[e] == kPad ? -1 : row_of[sel[e]];

  // (3a) a new round.  PB-LRU: the current bucket advances one position; what
  //      is left in the bucket about to be reused is folded into the cold bucket.
  //      (Exact LRU has no buckets; its ring stays empty.)
  g.round++;
  g.cur = (g.cur + 1) % o->B;
  if (!o->exact()) {
    for (uint32_t s : g.ring[g.cur]) {
      g.cold.insert(s);
      g.cls[s] = kCold;
    }
    g.ring[g.cur].clear();
  }

  // (3b) hits: the slot is accessed in this round (PB-LRU: it moves into the
  //      current bucket; exact LRU: its timestamp becomes this round).
  for (uint32_t a : uniq)
    if (g.where[a].tier == kOnGpu) touch(*o, g, g.where[a].slot);

  // (4) victims: free slots, then the cold bucket, then the ring from oldest
  //     (cur+1) to newest (cur-1); never the current bucket; lowest slot first.
  std::vector<uint32_t> victims;
  std::vector<int> victim_class;
  auto take = [&](const std::set<uint32_t> &from, int label) {
    for (uint32_t s : from) {
      if (victims.size() == M) return;
      victims.push_back(s);
      victim_class.push_back(label);
    }
  };
  take(g.free_slots, kFree);
  if (o->exact()) {
    // exact LRU: the oldest timestamp first, ties to the lowest slot; a slot
    // stamped in this round (a hit) is never taken
    for (const auto &ts : g.by_age) {
      if (victims.size() == M || ts.first == g.round) break;
      victims.push_back(ts.second);
      victim_class.push_back(kCold);
    }
  } else {
    take(g.cold, kCold);
    for (uint32_t d = 1; d < o->B; ++d) take(g.ring[(g.cur + d) % o->B], (int)((g.cur + d) % o->B));
  }

  if (victims.size() != M) return kInternal;

  // host slots for write-backs: the j-th lowest host slot free before the step
  std::vector<uint32_t> wb_host;
  for (uint32_t hs : g.host_free) {
    if (wb_host.size() == writebacks_needed) break;
    wb_host.push_back(hs);
  }

  // (5) move the data first: victim i (if it holds data) is written back to
  //     the host, then miss i is filled into it; then the map is updated.
  std::vector<uint32_t> released_host;
  size_t wb = 0;
  uint64_t n_free = 0, n_cold = 0, n_ring = 0;
  for (size_t i = 0; i < M; ++i) {
    const uint32_t v = victims[i];
    const uint32_t a = misses[i];
    const uint32_t src_host = g.where[a].slot;
    const uint32_t prev_owner = g.owner[v];
    if (victim_class[i] == kFree) ++n_free;
    else if (victim_class[i] == kCold) ++n_cold;
    else ++n_ring;
    if (prev_owner != kNone) {
      if (wb >= wb_host.size()) return kInternal;
      const uint32_t hs = wb_host[wb++];
      std::memcpy(&g.host_pool[(size_t)hs * sb], &g.gpu_pool[(size_t)v * sb], sb);
      g.host_free.erase(hs);
      g.host_owner[hs] = prev_owner;
      g.where[prev_owner] = Location{kOnHost, hs};
    }
    std::memcpy(&g.gpu_pool[(size_t)v * sb], &g.host_pool[(size_t)src_host * sb], sb);
    g.where[a] = Location{kOnGpu, v};
    g.owner[v] = a;
    touch(*o, g, v);
    released_host.push_back(src_host);
  }
  for (uint32_t hs : released_host) {
    g.host_free.insert(hs);
    g.host_owner[hs] = kNone;
  }

  // (6) gather through the committed map: out[j][u] = row j of uniq[u]'s slot.
  for (uint32_t j = 0; j < g.layers; ++j)
    for (size_t u = 0; u < uniq.size(); ++u) {
      const Location loc = g.where[uniq[u]];
      const std::vector<uint8_t> &pool = loc.tier == kOnGpu ? g.gpu_pool : g.host_pool;  // host: bypassed
      std::memcpy(out + ((size_t)j * out_cap + u) * o->row_bytes,
                  &pool[(size_t)loc.slot * sb + (size_t)j * o->row_bytes], o->row_bytes);
    }

  g.last_victims = victims;
  g.last_wb_host = wb_host;
  g.last_victim_class = victim_class;
  g.last_bypassed = bypassed.size();
  if (counters) {
    counters[0] = uniq.size();
    counters[1] = hits;
    counters[2] = M + bypassed.size();
    counters[3] = n_free;
    counters[4] = n_cold;
    counters[5] = n_ring;
    counters[6] = wb;
    counters[7] = (uint64_t)uniq.size() * g.layers;
    counters[8] = bypassed.size();
  }
  return kOk;
}

// Last step's decisions of group gi; returns the number of victims.
uint32_t orc_last_decisions(void *h, uint32_t gi, uint32_t *victims, int32_t *victim_class,
                            uint32_t *wb_host, uint32_t *n_wb) {
  Oracle *o = static_cast<Oracle *>(h);
  const Group &g = o->groups[gi];
  if (victims) std::copy(g.last_victims.begin(), g.last_victims.end(), victims);
  if (victim_class) std::copy(g.last_victim_class.begin(), g.last_victim_class.end(), victim_class);
  if (wb_host) std::copy(g.last_wb_host.begin(), g.last_wb_host.end(), wb_host);
  if (n_wb) *n_wb = (uint32_t)g.last_wb_host.size();
  return (uint32_t)g.last_victims.size();
}

// State of group gi.  tier/slot: [max_logical]; cls/owner: [S]; host_free: [H] (1 = free).
void orc_export(void *h, uint32_t gi, uint8_t *tier, uint32_t *slot, int32_t *cls,
                uint32_t *owner, uint8_t *host_free, uint32_t *host_owner, uint32_t *cur) {
  Oracle *o = static_cast<Oracle *>(h);
  const Group &g = o->groups[gi];
  for (uint32_t a = 0; a < o->max_logical; ++a) {
    if (tier) tier[a] = g.where[a].tier;
    if (slot) slot[a] = g.where[a].tier == kUnallocated ? 0 : g.where[a].slot;
  }
  if (cls) std::copy(g.cls.begin(), g.cls.end(), cls);
  if (owner) std::copy(g.owner.begin(), g.owner.end(), owner);
  if (host_free) {
    std::memset(host_free, 0, o->H);
    for (uint32_t hs : g.host_free) host_free[hs] = 1;
  }
  if (host_owner) std::copy(g.host_owner.begin(), g.host_owner.end(), host_owner);
  if (cur) *cur = g.cur;
}

// Timestamps of group gi's GPU slots ([S]: round of the last access, kNone if
// free) and its round count.
void orc_export_stamps(void *h, uint32_t gi, uint32_t *stamp, uint32_t *round) {
  Oracle *o = static_cast<Oracle *>(h);
  const Group &g = o->groups[gi];
  if (stamp) std::copy(g.stamp.begin(), g.stamp.end(), stamp);
  if (round) *round = g.round;
}

const uint8_t *orc_gpu_pool(void *h, uint32_t gi) {
  return static_cast<Oracle *>(h)->groups[gi].gpu_pool.data();
}
const uint8_t *orc_host_pool(void *h, uint32_t gi) {
  return static_cast<Oracle *>(h)->groups[gi].host_pool.data();
}

// ---------------------------------------------------------------------------
// Exact LRU companion (hit rate only).  The pages' baseline policy keeps one
// timestamp per slot and chooses victims by scanning for the oldest (§3
// "PB-LRU", first paragraph; §4 compares hit rates).  Here: a timestamp per
// GPU slot = the last round it was accessed (hit or filled); victims are free
// slots (lowest first), then the smallest timestamp, ties to the lowest slot.
// It keeps its own placement, so only hit/miss counts are comparable.

namespace {
struct LruGroup {
  std::vector<int64_t> where;  // [max_logical]: GPU slot, -1 on host, -2 unallocated
  std::vector<uint64_t> stamp; // [S]
  std::vector<uint32_t> owner; // [S]
  std::set<uint32_t> free_slots;
  std::set<std::pair<uint64_t, uint32_t>> by_age;  // (stamp, slot) of occupied slots
  uint64_t round = 0;
};
struct Lru {
  uint32_t S = 0, max_logical = 0, next_logical = 0;
  std::vector<LruGroup> groups;
};
}  // namespace

void *orc_lru_create(uint32_t n_groups, uint32_t S, uint32_t max_logical) {
  Lru *l = new Lru;
  l->S = S;
  l->max_logical = max_logical;
  l->groups.resize(n_groups);
  for (LruGroup &g : l->groups) {
    g.where.assign(max_logical, -2);
    g.stamp.assign(S, 0);
    g.owner.assign(S, kNone);
    for (uint32_t s = 0; s < S; ++s) g.free_slots.insert(s);
  }
  return l;
}

void orc_lru_destroy(void *h) { delete static_cast<Lru *>(h); }

int orc_lru_alloc(void *h, uint32_t n, uint32_t *base_out) {
  Lru *l = static_cast<Lru *>(h);
  if ((uint64_t)l->next_logical + n > l->max_logical) return kCapacity;
  const uint32_t base = l->next_logical;
  for (LruGroup &g : l->groups)
    for (uint32_t i = 0; i < n; ++i) {
      const uint32_t a = base + i;
      if (!g.free_slots.empty()) {
        uint32_t s = *g.free_slots.begin();
        g.free_slots.erase(s);
        g.stamp[s] = g.round;
        g.owner[s] = a;
        g.by_age.insert({g.round, s});
        g.where[a] = s;
      } else {
        g.where[a] = -1;
      }
    }
  l->next_logical = base + n;
  *base_out = base;
  return kOk;
}

int orc_lru_free(void *h, uint32_t base, uint32_t n) {
  Lru *l = static_cast<Lru *>(h);
  for (LruGroup &g : l->groups)
    for (uint32_t i = 0; i < n; ++i) {
      const int64_t w = g.where[base + i];
      if (w >= 0) {
        g.by_age.erase({g.stamp[w], (uint32_t)w});
        g.free_slots.insert((uint32_t)w);
        g.owner[w] = kNone;
      }
      g.where[base + i] = -2;
    }
  return kOk;
}

// Returns kOk and adds (uniq, hits) to acc[0], acc[1].
int orc_lru_step(void *h, uint32_t gi, const uint32_t *sel, size_t n_entries, uint64_t *acc) {
  Lru *l = static_cast<Lru *>(h);
  LruGroup &g = l->groups[gi];
  g.round++;
  std::unordered_map<uint32_t, char> seen;
  std::vector<uint32_t> uniq;
  for (size_t e = 0; e < n_entries; ++e) {
    const uint32_t a = sel[e];
    if (a == kPad) continue;
    if (a >= l->max_logical || g.where[a] == -2) return kUnmapped;
    if (seen.emplace(a, 1).second) uniq.push_back(a);
  }
  uint64_t hits = 0;
  std::vector<uint32_t> misses;
  for (uint32_t a : uniq) {
    const int64_t w = g.where[a];
    if (w >= 0) {
      ++hits;
      g.by_age.erase({g.stamp[w], (uint32_t)w});
      g.stamp[w] = g.round;
      g.by_age.insert({g.round, (uint32_t)w});
    } else {
      misses.push_back(a);
    }
  }
  for (uint32_t a : misses) {
    uint32_t s;
    if (!g.free_slots.empty()) {
      s = *g.free_slots.begin();
      g.free_slots.erase(s);
    } else {
      if (g.by_age.empty() || g.by_age.begin()->first == g.round) return kCapacity;
      s = g.by_age.begin()->second;
      g.by_age.erase(g.by_age.begin());
      g.where[g.owner[s]] = -1;
    }
    g.stamp[s] = g.round;
    g.owner[s] = a;
    g.by_age.insert({g.round, s});
    g.where[a] = s;
  }
  acc[0] += uniq.size();
  acc[1] += hits;
  return kOk;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// TP mode, emulated (§2 "Unified logical addresses", TP paragraph): address t
// belongs to partition t mod P (P partitions stand in for P GPUs).  Each
// partition is a DP residency (the code above) over its own addresses, with
// local ids t / P.  Each rank r also caches, per group, copies of the remote
// rows (t mod P != r) its steps selected: PB-LRU over the buffer's own slots and
// ring, a victim's copy is dropped (the owner keeps the entry), and a missing
// row is fetched from its owner's GPU slot, where the owner's step has just made
// it resident.

namespace {
struct Buffer {  // one rank's local buffer for one group
  uint32_t layers = 0;
  std::vector<int64_t> where;            // [max_logical]: buffer slot, or -1
  std::vector<int> cls;                  // [slots]
  std::vector<uint32_t> owner;           // [slots]
  std::set<uint32_t> free_slots, cold;
  std::vector<std::set<uint32_t>> ring;  // [B]
  uint32_t cur = 0;
  std::vector<uint8_t> pool;             // [slots][layers][row_bytes]
  std::vector<uint32_t> last_victims;
};

struct Tp {
  uint32_t P = 0, slots = 0, row_bytes = 0, n_groups = 0, max_logical = 0, B = 0;
  std::vector<uint32_t> layers;
  std::vector<Oracle *> parts;              // [P]
  std::vector<std::vector<Buffer>> buf;     // [P ranks][G]
  uint32_t next_logical = 0;
};

void buffer_to_current(Buffer &b, uint32_t s) {
  int c = b.cls[s];
  if (c == kFree) b.free_slots.erase(s);
  else if (c == kCold) b.cold.erase(s);
  else b.ring[(size_t)c].erase(s);
  b.ring[b.cur].insert(s);
  b.cls[s] = (int)b.cur;
}

// The rows of partition p among global addresses [base, base + n), per group, as
// the partition's alloc wants them (its local ids are consecutive).
std::vector<uint8_t> partition_rows(const Tp &t, uint32_t p, uint32_t base, uint32_t n,
                                    const uint8_t *rows, uint32_t *n_p) {
  std::vector<uint8_t> out;
  uint32_t cnt = 0;
  for (uint32_t a = base; a < base + n; ++a)
    if (a % t.P == p) ++cnt;
  size_t group_off = 0;
  for (uint32_t g = 0; g < t.n_groups; ++g) {
    const size_t sb = (size_t)t.layers[g] * t.row_bytes;
    for (uint32_t a = base; a < base + n; ++a)
      if (a % t.P == p) {
        const uint8_t *src = rows + group_off + (size_t)(a - base) * sb;
        out.insert(out.end(), src, src + sb);
      }
    group_off += (size_t)n * sb;
  }
  *n_p = cnt;
  return out;
}
}  // namespace

extern "C" {

void *orc_tp_create(uint32_t row_bytes, uint32_t n_groups, const uint32_t *layers, uint32_t P,
                    uint32_t S, uint32_t H, uint32_t B, uint32_t max_logical, uint32_t slots) {
  if (!P || !slots || !max_logical) return nullptr;
  Tp *t = new Tp;
  t->P = P;
  t->slots = slots;
  t->row_bytes = row_bytes;
  t->n_groups = n_groups;
  t->max_logical = max_logical;
  t->B = B;
  t->layers.assign(layers, layers + n_groups);
  const uint32_t local_max = (max_logical + P - 1) / P;
  for (uint32_t p = 0; p < P; ++p) {
    void *o = orc_create2(row_bytes, n_groups, layers, S, H, B, local_max, 0);
    if (!o) {
      for (Oracle *x : t->parts) delete x;
      delete t;
      return nullptr;
    }
    t->parts.push_back(static_cast<Oracle *>(o));
  }
  t->buf.resize(P);
  for (uint32_t r = 0; r < P; ++r) {
    t->buf[r].resize(n_groups);
    for (uint32_t g = 0; g < n_groups; ++g) {
      Buffer &b = t->buf[r][g];
      b.layers = layers[g];
      b.where.assign(max_logical, -1);
      b.cls.assign(slots, kFree);
      b.owner.assign(slots, kNone);
      for (uint32_t s = 0; s < slots; ++s) b.free_slots.insert(s);
      b.ring.assign(B, std::set<uint32_t>{});
      b.pool.assign((size_t)slots * layers[g] * row_bytes, 0);
    }
  }
  return t;
}

void orc_tp_destroy(void *h) {
  Tp *t = static_cast<Tp *>(h);
  for (Oracle *o : t->parts) delete o;
  delete t;
}

// rows: per group, [n][layers_g][row_bytes] in global address order.
int orc_tp_alloc(void *h, uint32_t n, const uint8_t *rows, uint32_t *base_out) {
  Tp *t = static_cast<Tp *>(h);
  if (!base_out || (n && !rows)) return kInvalidArg;
  if ((uint64_t)t->next_logical + n > t->max_logical) return kCapacity;
  const uint32_t base = t->next_logical;
  for (uint32_t p = 0; p < t->P; ++p) {
    uint32_t n_p = 0;
    std::vector<uint8_t> r = partition_rows(*t, p, base, n, rows, &n_p);
    uint32_t local_base = 0;
    const int rc = orc_alloc(t->parts[p], n_p, n_p ? r.data() : nullptr, &local_base);
    if (rc) return rc;  // (earlier partitions keep their part: TP errors are not atomic)
  }
  t->next_logical = base + n;
  *base_out = base;
  return kOk;
}

int orc_tp_free(void *h, uint32_t base, uint32_t n) {
  Tp *t = static_cast<Tp *>(h);
  if ((uint64_t)base + n > t->max_logical) return kInvalidArg;
  for (uint32_t p = 0; p < t->P; ++p) {
    // partition p's addresses in the range are consecutive local ids
    uint32_t first = base, cnt = 0;
    while (first < base + n && first % t->P != p) ++first;
    for (uint32_t a = first; a < base + n; a += t->P) ++cnt;
    if (cnt) {
      const int rc = orc_free(t->parts[p], first / t->P, cnt);
      if (rc) return rc;
    }
  }
  for (auto &per_rank : t->buf)  // buffered copies of freed addresses are dropped
    for (Buffer &b : per_rank)
      for (uint32_t a = base; a < base + n; ++a)
        if (b.where[a] >= 0) {
          const uint32_t s = (uint32_t)b.where[a];
          int c = b.cls[s];
          if (c == kCold) b.cold.erase(s);
          else if (c != kFree) b.ring[(size_t)c].erase(s);
          b.free_slots.insert(s);
          b.cls[s] = kFree;
          b.owner[s] = kNone;
          b.where[a] = -1;
        }
  return kOk;
}

// One TP step of group gi.  For partition (and rank) r: local_out[r], local_entry_row[r],
// local_req_off[r] are partition r's DP step on the entries it owns (the others as pads,
// addresses as local ids); remote_out[r], remote_entry_row[r], remote_req_off[r] are rank
// r's buffer step on the entries it does not own.  counters (optional) [P][2][9]: the DP
// counters of partition r, then the buffer's (uniq, hits, misses, victims from free, cold,
// ring, 0, rows gathered, 0).
int orc_tp_step_group(void *h, uint32_t gi, const uint32_t *sel, uint32_t n_req, uint32_t q,
                      uint32_t k, uint8_t *const *local_out, uint8_t *const *remote_out,
                      uint32_t out_cap, int32_t *const *local_entry_row,
                      int32_t *const *local_req_off, int32_t *const *remote_entry_row,
                      int32_t *const *remote_req_off, uint64_t *counters) {
  Tp *t = static_cast<Tp *>(h);
  if (gi >= t->n_groups) return kInvalidArg;
  const size_t E = (size_t)n_req * q * k;
  const uint32_t P = t->P;
  // (1) every partition steps on the entries it owns
  std::vector<uint32_t> part_sel(E);
  for (uint32_t p = 0; p < P; ++p) {
    for (size_t e = 0; e < E; ++e)
      part_sel[e] = (sel[e] != kPad && sel[e] % P == p) ? sel[e] / P : kPad;
    const int rc = orc_step_group(t->parts[p], gi, part_sel.data(), n_req, q, k, local_out[p],
                                  out_cap, local_entry_row[p], local_req_off[p],
                                  counters ? counters + (size_t)p * 18 : nullptr);
    if (rc) return rc;
  }
  // (2) every rank's buffer takes the entries it does not own
  for (uint32_t r = 0; r < P; ++r) {
    Buffer &b = t->buf[r][gi];
    const size_t sb = (size_t)b.layers * t->row_bytes;
    std::vector<uint32_t> uniq;
    std::unordered_map<uint32_t, int32_t> row_of;
    int32_t *er = remote_entry_row[r];
    int32_t *ro = remote_req_off[r];
    for (uint32_t rq = 0; rq < n_req; ++rq) {
      ro[rq] = (int32_t)uniq.size();
      for (size_t e = (size_t)rq * q * k; e < (size_t)(rq + 1) * q * k; ++e) {
        const uint32_t a = sel[e];
        if (a == kPad || a % P == r) continue;
        if (row_of.find(a) == row_of.end()) {
          row_of.emplace(a, (int32_t)uniq.size());
          uniq.push_back(a);
        }
      }
    }
    ro[n_req] = (int32_t)uniq.size();
    for (size_t e = 0; e < E; ++e)
      er[e] = (sel[e] == kPad || sel[e] % P == r) ? -1 : row_of[sel[e]];
    std::vector<uint32_t> misses;
    size_t hits = 0;
    for (uint32_t a : uniq) {
      if (b.where[a] >= 0) ++hits;
      else misses.push_back(a);
    }
    if (uniq.size() > out_cap || misses.size() > t->slots - hits) return kCapacity;
    // rotate, then hits into the current bucket
    b.cur = (b.cur + 1) % t->B;
    for (uint32_t s : b.ring[b.cur]) {
      b.cold.insert(s);
      b.cls[s] = kCold;
    }
    b.ring[b.cur].clear();
    for (uint32_t a : uniq)
      if (b.where[a] >= 0) buffer_to_current(b, (uint32_t)b.where[a]);
    // victims: free, cold, ring oldest -> newest, lowest slot first
    std::vector<uint32_t> victims;
    std::vector<int> vcls;
    auto take = [&](const std::set<uint32_t> &from, int label) {
      for (uint32_t s : from) {
        if (victims.size() == misses.size()) return;
        victims.push_back(s);
        vcls.push_back(label);
      }
    };
    take(b.free_slots, kFree);
    take(b.cold, kCold);
    for (uint32_t d = 1; d < t->B; ++d) take(b.ring[(b.cur + d) % t->B], (int)((b.cur + d) % t->B));
    if (victims.size() != misses.size()) return kInternal;
    uint64_t n_free = 0, n_cold = 0;
    for (size_t i = 0; i < misses.size(); ++i) {
      const uint32_t v = victims[i], a = misses[i];
      if (vcls[i] == kFree) ++n_free;
      else if (vcls[i] == kCold) ++n_cold;
      if (b.owner[v] != kNone) b.where[b.owner[v]] = -1;  // the copy is dropped
      // fetch from the owner partition's GPU slot (resident after its step)
      const Oracle *o = t->parts[a % P];
      const Group &og = o->groups[gi];
      const Location loc = og.where[a / P];
      if (loc.tier != kOnGpu) return kInternal;
      std::memcpy(&b.pool[(size_t)v * sb], &og.gpu_pool[(size_t)loc.slot * sb], sb);
      b.where[a] = v;
      b.owner[v] = a;
      buffer_to_current(b, v);
    }
    b.last_victims = victims;
    for (uint32_t j = 0; j < b.layers; ++j)
      for (size_t u = 0; u < uniq.size(); ++u)
        std::memcpy(remote_out[r] + ((size_t)j * out_cap + u) * t->row_bytes,
                    &b.pool[(size_t)b.where[uniq[u]] * sb + (size_t)j * t->row_bytes], t->row_bytes);
    if (counters) {
      uint64_t *c = counters + (size_t)r * 18 + 9;
      c[0] = uniq.size();
      c[1] = hits;
      c[2] = misses.size();
      c[3] = n_free;
      c[4] = n_cold;
      c[5] = misses.size() - n_free - n_cold;
      c[6] = 0;
      c[7] = (uint64_t)uniq.size() * b.layers;
      c[8] = 0;
    }
  }
  return kOk;
}

// Rank r's buffer of group gi: where [max_logical] (slot or -1), owner/cls [slots], cur;
// returns the number of victims of its last step (copied to victims if given).
uint32_t orc_tp_buffer(void *h, uint32_t r, uint32_t gi, int64_t *where, uint32_t *owner,
                       int32_t *cls, uint32_t *cur, uint32_t *victims) {
  Tp *t = static_cast<Tp *>(h);
  const Buffer &b = t->buf[r][gi];
  if (where) std::copy(b.where.begin(), b.where.end(), where);
  if (owner) std::copy(b.owner.begin(), b.owner.end(), owner);
  if (cls) std::copy(b.cls.begin(), b.cls.end(), cls);
  if (cur) *cur = b.cur;
  if (victims) std::copy(b.last_victims.begin(), b.last_victims.end(), victims);
  return (uint32_t)b.last_victims.size();
}

// Partition p's oracle handle (for its export / pools).
void *orc_tp_partition(void *h, uint32_t p) { return static_cast<Tp *>(h)->parts[p]; }

}  // extern "C"
