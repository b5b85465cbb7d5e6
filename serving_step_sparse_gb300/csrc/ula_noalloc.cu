// ula_dedup_noalloc: first-occurrence dedup of a selection with no allocation.
//
// Who this is for: code that must not call cudaMalloc at the point where it
// dedups -- for example a serving engine that reserved nearly all HBM for its
// KV pools at start-up (an allocation would fail or fragment), or a hot path
// that cannot afford cudaMalloc's implicit device synchronisation and
// unbounded latency.  Such callers pass device inputs and outputs only; the
// scratch lives in a fixed file-scope device array that this library carries
// (about 1.3 MB, held on every device that loads the library until the process
// exits).
//
// The result is the same as the dedup inside ula_step_group: unique addresses
// in order of first occurrence, and for each entry the row of its address
// (-1 for pads).  Instead of that path's table indexed by logical address, the
// scratch here is an open-addressing hash table sized by the entry count, so
// addresses may be any 32-bit value except the pad marker.
#include <mutex>

#include "ula.h"

namespace {

constexpr uint32_t kMaxEntries = ULA_NOALLOC_MAX_ENTRIES;
constexpr uint32_t kTable = 2 * kMaxEntries;  // load factor <= 1/2: probing always ends
constexpr uint32_t kEmpty = 0xFFFFFFFFu;
constexpr int kThreads = 256;
constexpr uint32_t kMaxBlocks = (kMaxEntries + kThreads - 1) / kThreads;

// The shared scratch.  Layout (32-bit words):
//   keys[kTable]    address stored in each hash slot (kEmpty = unused)
//   first[kTable]   smallest entry index seen for the slot's address
//   row[kTable]     unique row of the slot's address
//   blk[kMaxBlocks + 1]  per-block first-occurrence counts, then their offsets
struct Scratch {
  uint32_t keys[kTable];
  uint32_t first[kTable];
  uint32_t row[kTable];
  uint32_t blk[kMaxBlocks + 1];
};

__device__ __align__(256) Scratch g_dedup_scratch;

// A call uses the first 2^bits slots of the table, the smallest power of two at or
// above 2n (load factor <= 1/2 whatever n is), so that it clears and probes no more
// than its size needs.
constexpr uint32_t kTableBits = 17;
static_assert(kTable == (1u << kTableBits), "table of 2^17 slots");

uint32_t table_bits(uint32_t n) {
  uint32_t bits = 1;
  while (bits < kTableBits && (1u << bits) < 2 * n) ++bits;
  return bits;
}

__device__ __forceinline__ uint32_t hash_slot(uint32_t a, uint32_t bits) {
  // multiplicative hashing (Knuth), top bits select the slot
  return (a * 2654435761u) >> (32 - bits);
}

__device__ __forceinline__ uint32_t find_slot(const Scratch *s, uint32_t a, uint32_t bits) {
  const uint32_t mask = (1u << bits) - 1;
  uint32_t h = hash_slot(a, bits);
  for (uint32_t i = 0; i <= mask; ++i) {
    if (s->keys[h] == a) return h;
    h = (h + 1) & mask;
  }
  return kEmpty;
}

__global__ void k_clear(Scratch *s, uint32_t bits) {
  const uint32_t size = 1u << bits;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < size; i += gridDim.x * blockDim.x) {
    s->keys[i] = kEmpty;
    s->first[i] = kEmpty;
  }
}

__global__ void k_insert(Scratch *s, const uint32_t *sel, uint32_t n, uint32_t bits) {
  const uint32_t e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  const uint32_t a = sel[e];
  if (a == ULA_ADDR_PAD) return;
  const uint32_t mask = (1u << bits) - 1;
  uint32_t h = hash_slot(a, bits);
  for (uint32_t i = 0; i <= mask; ++i) {
    const uint32_t k = atomicCAS(&s->keys[h], kEmpty, a);
    if (k == kEmpty || k == a) {
      atomicMin(&s->first[h], e);
      return;
    }
    h = (h + 1) & mask;
  }
}

__device__ __forceinline__ uint32_t is_first(const Scratch *s, const uint32_t *sel, uint32_t n,
                                             uint32_t bits, uint32_t e, uint32_t *slot) {
  *slot = kEmpty;
  if (e >= n || sel[e] == ULA_ADDR_PAD) return 0;
  *slot = find_slot(s, sel[e], bits);
  return *slot != kEmpty && s->first[*slot] == e ? 1u : 0u;
}

__device__ __forceinline__ uint32_t warp_incl(uint32_t v) {
  const uint32_t lane = threadIdx.x & 31;
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= (uint32_t)d) v += t;
  }
  return v;
}

// per-block counts of first occurrences
__global__ void __launch_bounds__(kThreads) k_count(Scratch *s, const uint32_t *sel, uint32_t n,
                                                    uint32_t bits) {
  uint32_t slot;
  const uint32_t f = is_first(s, sel, n, bits, blockIdx.x * blockDim.x + threadIdx.x, &slot);
  const uint32_t c = __syncthreads_count(f);
  if (threadIdx.x == 0) s->blk[blockIdx.x] = c;
}

// exclusive offsets of the blocks (nblk <= kMaxBlocks <= blockDim.x); total to *n_uniq
__global__ void __launch_bounds__(kThreads) k_offsets(Scratch *s, uint32_t nblk, uint32_t *n_uniq) {
  __shared__ uint32_t wsum[kThreads / 32];
  const uint32_t t = threadIdx.x;
  uint32_t acc = 0;
  for (uint32_t base = 0; base < nblk; base += kThreads) {
    const uint32_t i = base + t;
    const uint32_t v = i < nblk ? s->blk[i] : 0u;
    const uint32_t inc = warp_incl(v);
    if ((t & 31) == 31) wsum[t >> 5] = inc;
    __syncthreads();
    uint32_t before = 0;
    for (uint32_t w = 0; w < (t >> 5); ++w) before += wsum[w];
    uint32_t chunk = 0;
    for (uint32_t w = 0; w < kThreads / 32; ++w) chunk += wsum[w];
    __syncthreads();
    if (i < nblk) s->blk[i] = acc + before + inc - v;
    acc += chunk;
  }
  if (t == 0) *n_uniq = acc;
}

__global__ void __launch_bounds__(kThreads) k_emit(Scratch *s, const uint32_t *sel, uint32_t n,
                                                   uint32_t bits, uint32_t *uniq) {
  __shared__ uint32_t wsum[kThreads / 32];
  const uint32_t e = blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t slot;
  const uint32_t f = is_first(s, sel, n, bits, e, &slot);
  const uint32_t inc = warp_incl(f);
  if ((threadIdx.x & 31) == 31) wsum[threadIdx.x >> 5] = inc;
  __syncthreads();
  uint32_t pos = s->blk[blockIdx.x] + inc - f;
  for (uint32_t w = 0; w < (threadIdx.x >> 5); ++w) pos += wsum[w];
  if (f) {
    uniq[pos] = sel[e];
    s->row[slot] = pos;
  }
}

__global__ void k_rows(const Scratch *s, const uint32_t *sel, uint32_t n, uint32_t bits,
                       int32_t *entry_row) {
  const uint32_t e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  const uint32_t a = sel[e];
  if (a == ULA_ADDR_PAD) {
    entry_row[e] = -1;
    return;
  }
  const uint32_t h = find_slot(s, a, bits);
  entry_row[e] = h == kEmpty ? -1 : (int32_t)s->row[h];
}

// Device address of the scratch, looked up once per device (with that device current).
// A device reset (cudaDeviceReset) reloads the library's device code, possibly at
// another address: the cached address is then stale, and the entry point must not be
// used again in this process.
constexpr int kMaxDevices = 64;
std::mutex g_lock;
Scratch *g_addr[kMaxDevices] = {};

int scratch_for_current_device(Scratch **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ULA_ERR_CUDA;
  std::lock_guard<std::mutex> guard(g_lock);
  if (!g_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dedup_scratch) != cudaSuccess || !p) {
      cudaGetLastError();  // (this call's own error)
      return ULA_ERR_CUDA;
    }
    g_addr[dev] = static_cast<Scratch *>(p);
  }
  *out = g_addr[dev];
  return ULA_OK;
}

// One launch; its own status (not an earlier error left on this thread).
template <typename... Args>
cudaError_t launch(void (*kernel)(Args...), uint32_t grid, uint32_t block, cudaStream_t st,
                   Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.stream = st;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

extern "C" int ula_dedup_noalloc(const uint32_t *d_sel, uint32_t n, uint32_t *d_uniq,
                                 int32_t *d_entry_row, uint32_t *d_n_uniq, void *stream) {
  if (n > kMaxEntries) return ULA_ERR_CAPACITY;
  if (!d_n_uniq || (n && (!d_sel || !d_uniq || !d_entry_row))) return ULA_ERR_INVALID_ARG;
  Scratch *s = nullptr;
  int rc = scratch_for_current_device(&s);
  if (rc != ULA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint32_t nblk = (n + kThreads - 1) / kThreads;
  const uint32_t bits = table_bits(n);
  const uint32_t clear_blocks = ((1u << bits) + 255) / 256;
  cudaError_t e = launch(k_clear, clear_blocks < 128 ? clear_blocks : 128, 256, st, s, bits);
  if (e == cudaSuccess && nblk) e = launch(k_insert, nblk, kThreads, st, s, d_sel, n, bits);
  if (e == cudaSuccess && nblk) e = launch(k_count, nblk, kThreads, st, s, d_sel, n, bits);
  if (e == cudaSuccess) e = launch(k_offsets, 1, kThreads, st, s, nblk, d_n_uniq);
  if (e == cudaSuccess && nblk) e = launch(k_emit, nblk, kThreads, st, s, d_sel, n, bits, d_uniq);
  if (e == cudaSuccess && nblk) e = launch(k_rows, nblk, kThreads, st, static_cast<const Scratch *>(s), d_sel, n, bits, d_entry_row);
  return e == cudaSuccess ? ULA_OK : ULA_ERR_CUDA;
}
