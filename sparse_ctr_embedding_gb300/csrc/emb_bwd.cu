// Backward: duplicate-key gradient reduction + the fused sparse update
// (element-wise Adagrad, or FTRL-Proximal).
//
// Tencent PCG DataFun talk, "计算优化": one backward kernel updates every
// feature of the unified table.  JD ads article, 3.2.1: Adagrad keeps a
// per-parameter sum of squared gradients, updates element-wise, and leaves
// features that are absent from the batch untouched; FTRL is the other
// sparse optimizer it names.
//
// Pipeline (all on the caller's stream, no host synchronisation):
//  0. placement the bag lengths, transposed to slot-major order and scanned,
//               give every bag's first pair position: each slot's pairs
//               form one region of the pair arrays.
//  1. expand    (without a recording forward) one warp per bag: probe each
//               key; write the pair (internal row, bag) of every occurrence
//               at its placed position (row = n_rows for a miss, which sorts
//               last in its slot) and, for mean, 1/L per bag.
//  2. sort      stable LSD radix sort of each region's pairs by the in-slot
//               row number (hand-written: per-tile digit counts, a
//               device-wide scan, then a stable scatter ranked with warp
//               match and staged in shared memory so every digit run is
//               written contiguously).  Rows are numbered slot-major, so the
//               sorted order walks one feature slot (one column block of
//               grad_out) at a time.
//  3. reduce    the sorted positions are cut into sub-chunks (128 or 256
//               positions, fewer for small batches) taken in order from a
//               counter by groups of G lanes.  Every run of equal rows
//               inside a sub-chunk ("piece") is summed in float32 with TwoSum
//               compensation, in sorted order (so in occurrence order: the
//               sort is stable).  A piece that is a whole segment (all
//               occurrences of its row) gets the update directly.  A piece
//               cut by a sub-chunk edge leaves a partial sum: the head piece
//               of a segment in slot A of its sub-chunk, later pieces in
//               slot B of theirs.
//  4. fold      (large batches) every block of 32 sub-chunks inside one
//               row's run has its slot-B partials summed into one.
//  5. fixup     one warp per segment that spans sub-chunks: A + B + B ...
//               (a folded block as one) in sub-chunk order (compensated,
//               then a fixed tree across the warp's lane groups), then the
//               update.
// No float atomics: every sum has a fixed order, so the step is bitwise
// reproducible.  The Adagrad arithmetic per element, in float32:
//   g = G;  acc += g * g;  w -= lr * g / (sqrt(acc) + eps)
// with sqrt and the quotient from the hardware reciprocal square root and
// fast division (a few ulp; see AdagradStep), half weights rounded to
// nearest-even on store.
#include <algorithm>
#include <cstdio>
#include <mutex>
#include <type_traits>
#include <utility>
#include <vector>

#include "emb_internal.cuh"

namespace emb {

emb_status check_batch(const emb_table* t, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                       int64_t nnz, int pool);
cudaError_t launch_forward(const emb_table* t, const long long* offsets, long long n_bags, const long long* keys,
                           long long nnz, int mean, float* out, unsigned* K, unsigned* V, float* scale,
                           const unsigned* dest, const unsigned* placed, unsigned long long* work, cudaStream_t st);

constexpr int kChunk = 256;                      // sorted positions per reduce sub-chunk (the largest batches)
constexpr int kMinChunk = 32;                    // the shortest sub-chunk (small batches)
constexpr size_t kLongChunkFrom = size_t(1) << 27;  // positions from which sub-chunks are kChunk long
constexpr unsigned kFoldChunks = 32;             // sub-chunks per fold block (fixup of long rows)
constexpr size_t kFoldFrom = size_t(1) << 24;     // positions from which the fold kernel runs
constexpr int kSortWarps = 8;
constexpr int kSortThreads = kSortWarps * 32;
constexpr int kSortItems = 16;                   // keys per lane per tile
constexpr int kSortTile = kSortThreads * kSortItems;
constexpr int kRadixBits = EMB_SORT_DIGIT_BITS;  // 7: 27-bit rows (100M) sort in 4 passes
constexpr int kDigits = 1 << kRadixBits;
constexpr int kScanThreads = 256;
constexpr int kScanItems = 16;
constexpr int kScanTile = kScanThreads * kScanItems;
constexpr unsigned kNoRow = 0xFFFFFFFFu;
constexpr unsigned kMagic = 0x454D4257u;  // "EMBW"

// Workspace header (first 256 bytes of the caller's workspace).
struct WsHeader {
  unsigned magic;
  unsigned nnz;
  unsigned n_bags;
  unsigned sorted_in_b;      // 1: sorted pairs are in buffer B
  unsigned miss_row;         // sentinel row of a miss (= n_rows)
  unsigned n_unique;         // filled by emb_bwd_unique_keys
  unsigned long long total;  // sum of the (clamped) bag lengths: nnz unless the offsets are malformed
  unsigned placed;           // 1: the clamped bags tile [0, nnz), pairs may be recorded
};

// One region of the sort: the pairs of one feature slot, or (the last region)
// pairs that are made absent.  Regions tile the positions [0, nnz) in order.
struct SortSeg {
  unsigned lo, hi;  // positions [lo, hi)
  unsigned tile0;   // first sort tile of the region (the entry after the last region: the tile count)
  unsigned rbase;   // first internal row of the slot
  unsigned cap;     // rows of the slot: in-slot row numbers are clamped to it, so misses sort last
  unsigned absent;  // 1: the first sort pass turns every pair of the region into an absent pair
  unsigned pad0, pad1;
};

static size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
  size_t hdr, kA, kB, vA, vB, scale, dest, sseg, treg, counts, partials, partA, partB, partC, folded, arow, zero, work,
      fwork, uniq, total;
  unsigned n_tiles_sort, n_regions, n_chunks, chunk, n_scan_partials, n_fold;
  int max_dim;
};

static WsLayout ws_layout(const emb_table* t, long long n_bags, long long nnz) {
  WsLayout L{};
  const size_t n = (size_t)std::max<long long>(nnz, 1);
  const size_t nb = (size_t)std::max<long long>(n_bags, 1);
  L.max_dim = t->st.max_dim;
  L.n_regions = (unsigned)t->st.n_slots + 1;  // one per slot, then the absent region
  // every region adds at most one partial tile
  L.n_tiles_sort = (unsigned)((n + kSortTile - 1) / kSortTile) + L.n_regions;
  // sub-chunk length: 256 positions from 2^27 positions up, else 128 (measured
  // per workload: at 282M positions 128 doubles the fixup, +0.6 ms; at 36M,
  // 6.5M and 4.5M positions it saves 0.07, 0.03 and 0.06 ms of reduce plus
  // fixup), halved down to 32 while that leaves fewer than about 64
  // sub-chunks per SM (a small batch then still spreads over every SM
  // instead of a few groups walking long sub-chunks in turn)
  L.chunk = n >= kLongChunkFrom ? kChunk : kChunk / 2;
  while (L.chunk > kMinChunk && n < (size_t)L.chunk * 64 * (size_t)sm_count()) L.chunk >>= 1;
  L.n_chunks = (unsigned)((n + L.chunk - 1) / L.chunk);
  const size_t n_counts = (size_t)kDigits * L.n_tiles_sort;
  const size_t scan_n = std::max(std::max(n_counts, n), nb);
  L.n_scan_partials = (unsigned)((scan_n + kScanTile - 1) / kScanTile);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o += align_up(std::max<size_t>(bytes, 1));
    return at;
  };
  L.hdr = take(sizeof(WsHeader));
  L.kA = take(n * 4);
  L.kB = take(n * 4);
  L.vA = take(n * 4);
  L.vB = take(n * 4);
  L.scale = take(nb * 4);
  L.dest = take(nb * 4);                                  // first position of each bag's pairs
  L.sseg = take((size_t)(L.n_regions + 1) * sizeof(SortSeg));
  L.treg = take((size_t)L.n_tiles_sort * 4);              // region of each sort tile
  L.counts = take(n_counts * 4);
  L.partials = take((size_t)(L.n_scan_partials + 1) * 4);
  L.partA = take((size_t)L.n_chunks * L.max_dim * 4);
  L.partB = take((size_t)L.n_chunks * L.max_dim * 4);
  L.n_fold = (L.n_chunks + kFoldChunks - 1) / kFoldChunks;
  L.partC = take((size_t)L.n_fold * L.max_dim * 4);   // folded partial of each block of kFoldChunks sub-chunks
  L.folded = take((size_t)L.n_fold * 4);
  L.arow = take((size_t)L.n_chunks * 4);
  L.zero = take((size_t)EMB_MAX_DIM * 4);  // a zero grad_out row (the widest lane group) for positions that add nothing
  L.work = take(sizeof(unsigned));        // sub-chunk counter of the reduce
  L.fwork = take(sizeof(unsigned long long));  // bag counter of the recording forward
  L.uniq = L.kA;  // emb_bwd_unique_keys reuses the buffer that is not holding the sorted keys
  L.total = o;
  return L;
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ------------------------------------------------------------------ 1. expand

// Unrecorded path: one warp per bag probes its keys and writes the pair
// (internal row, bag) of every occurrence at the bag's place in the slot-major
// order (dest, see placement below; row n_rows for a miss, which sorts last
// in its slot), and 1/L per bag for mean.
__global__ void __launch_bounds__(256) expand_kernel(TableView t, const long long* __restrict__ offsets,
                                                     long long n_bags, const long long* __restrict__ keys,
                                                     long long nnz, int mean, const unsigned* __restrict__ dest,
                                                     unsigned* __restrict__ K, unsigned* __restrict__ V,
                                                     float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const long long gw = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const unsigned S = (unsigned)t.n_slots;
  const unsigned long long B = (unsigned long long)n_bags / S;
  for (long long bag = gw; bag < n_bags; bag += nwarps) {
    const int s = (int)((unsigned)bag % S);
    long long start = offsets[bag], end = offsets[bag + 1];
    if (start < 0 || end > nnz || end < start || (bag == 0 && start != 0) || (bag == n_bags - 1 && end != nnz)) {
      if (lane == 0) atomicOr(t.flags, EMB_FLAG_BAD_OFFSETS);
      start = min(max(start, 0LL), nnz);
      end = min(max(end, start), nnz);
    }
    if (mean && lane == 0) scale[bag] = end > start ? 1.0f / (float)(end - start) : 0.f;
    const long long d0 = (long long)dest[(unsigned long long)s * B + (unsigned long long)bag / S] - start;
    for (long long i = start + lane; i < end; i += 32) {
      const long long k = keys[i];
      unsigned row = t.n_rows, ext;
      unsigned long long h;
      if (key_slot(k) != s) {
        atomicOr(t.flags, EMB_FLAG_SLOT_MISMATCH);
      } else if (!probe(t, k, &row, &ext, &h)) {
        row = t.n_rows;
      }
      const long long p = d0 + i;  // inside [0, nnz) unless the offsets are malformed
      if (p < nnz) {
        K[p] = row;
        V[p] = (unsigned)bag;
      }
    }
  }
}

// ------------------------------------------------------------------ 2. radix sort

// Lanes of the warp whose digit equals this lane's (invalid lanes form their
// own group), with one match instruction: measured 5.74 ms for the sort at
// 100M keys against 5.90 with one ballot per digit bit, 0.79 against 0.84
// at 100 slots x dim 32.
__device__ __forceinline__ unsigned warp_peers(unsigned d, bool valid) {
  return __match_any_sync(0xffffffffu, valid ? d : 0xFFFFFFFFu);
}

// Stable per-warp ranking over one tile: each warp walks its 32*kSortItems
// consecutive keys in order, 32 at a time; the lowest lane of each group of
// equal digits bumps the warp's counter for that digit.  Returns, per item,
// its rank among equal digits of this warp.
__device__ __forceinline__ void warp_rank(unsigned (&d)[kSortItems], unsigned (&rank)[kSortItems], bool (&valid)[kSortItems],
                                          unsigned* cnt /* this warp's kDigits counters */) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < kSortItems; ++r) {
    const unsigned peers = warp_peers(d[r], valid[r]);
    const int leader = __ffs(peers) - 1;
    unsigned base = 0;
    // one shared atomic per group (the counter's old value): successive
    // items' updates pipeline instead of chaining a load and a store
    if (valid[r] && lane == leader) base = atomicAdd(&cnt[d[r]], (unsigned)__popc(peers));
    base = __shfl_sync(0xffffffffu, base, leader);
    rank[r] = base + __popc(peers & lanemask_lt());
    __syncwarp();
  }
}

// The sort region of a tile: the largest r < n_regions with sg[r].tile0 <=
// tile, or n_regions for the spare tiles past the last region (the launch
// covers the most tiles any placement can need).
__device__ __forceinline__ unsigned region_of_tile(const SortSeg* __restrict__ sg, unsigned n_regions, unsigned tile) {
  if (tile >= sg[n_regions].tile0) return n_regions;
  unsigned lo = 0, hi = n_regions - 1;
  while (lo < hi) {
    const unsigned mid = (lo + hi + 1) >> 1;
    if (sg[mid].tile0 <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Digit of a row in its region: of the in-slot row number, clamped to the
// slot's row count so that misses (row n_rows) sort last; 0 in the absent region.
__device__ __forceinline__ unsigned region_digit(const SortSeg& g, unsigned k, int shift) {
  if (g.absent) return 0u;
  const unsigned in_slot = min(k - g.rbase, g.cap);  // k < rbase wraps high and clamps too
  return (in_slot >> shift) & (kDigits - 1);
}

// Digit counts of one tile of one region (the same keys the scatter kernel
// ranks), laid out region by region, digit-major within a region, so that
// one exclusive scan of the whole array gives every (tile, digit) its first
// output position and each region's output stays inside the region.  Each
// warp reads its 32*kSortItems keys 32 at a time (coalesced wherever the
// region starts) and adds each key with one shared atomic into the warp's
// own counters (measured: 5.38 ms for the three passes at 100M keys against
// 5.68 when the tile was staged in shared memory for runs of equal digits
// to be added at once).
__global__ void __launch_bounds__(kSortThreads) radix_count_kernel(const unsigned* __restrict__ keys,
                                                                   const SortSeg* __restrict__ sg,
                                                                   unsigned n_regions, int shift,
                                                                   unsigned* __restrict__ counts,
                                                                   const unsigned* __restrict__ tile_reg) {
  __shared__ unsigned cnt[kSortWarps][kDigits];
  __shared__ unsigned reg;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned tile = blockIdx.x;
  if (threadIdx.x == 0) reg = tile_reg ? tile_reg[tile] : region_of_tile(sg, n_regions, tile);
  for (int i = threadIdx.x; i < kSortWarps * kDigits; i += kSortThreads) (&cnt[0][0])[i] = 0;
  __syncthreads();
  const unsigned r = reg;
  if (r == n_regions) {  // a spare tile: zero counts in its own slice, after every region's
    for (int dg = threadIdx.x; dg < kDigits; dg += kSortThreads) counts[(size_t)kDigits * tile + dg] = 0;
    return;
  }
  const SortSeg g = sg[r];
  const unsigned nt = sg[r + 1].tile0 - g.tile0, lt = tile - g.tile0;
  const unsigned lo = g.lo + lt * kSortTile, hi = min(lo + kSortTile, g.hi);
  const unsigned wb = lo + (unsigned)w * 32u * kSortItems;
  unsigned kq[kSortItems];
#pragma unroll
  for (int q = 0; q < kSortItems; ++q) {
    const unsigned i = wb + q * 32 + lane;
    kq[q] = i < hi ? keys[i] : 0u;
  }
#pragma unroll
  for (int q = 0; q < kSortItems; ++q)
    if (wb + q * 32 + lane < hi) atomicAdd(&cnt[w][region_digit(g, kq[q], shift)], 1u);
  __syncthreads();
  for (int dg = threadIdx.x; dg < kDigits; dg += kSortThreads) {
    unsigned tot = 0;
#pragma unroll
    for (int ww = 0; ww < kSortWarps; ++ww) tot += cnt[ww][dg];
    counts[(size_t)kDigits * g.tile0 + (size_t)dg * nt + lt] = tot;
  }
}

// Block-wide exclusive scan of one value per thread.  sm needs 33 words; the
// block total is left in sm[32] for the caller.
__device__ __forceinline__ unsigned block_excl_scan(unsigned v, unsigned* sm) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int nw = (int)(blockDim.x >> 5);
  unsigned x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();  // sm may still be read by a previous call
  if (lane == 31) sm[w] = x;
  __syncthreads();
  if (w == 0) {
    unsigned t = lane < nw ? sm[lane] : 0;
    unsigned incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane < nw) sm[lane] = incl - t;
    if (lane == nw - 1) sm[32] = incl;
  }
  __syncthreads();
  return sm[w] + x - v;
}

// Stable scatter of one tile of one region by digit.  In the absent region
// every pair becomes (miss row, n_bags) as it is loaded.
__global__ void __launch_bounds__(kSortThreads, 3) radix_scatter_kernel(
    const unsigned* __restrict__ kin, const unsigned* __restrict__ vin, unsigned* __restrict__ kout,
    unsigned* __restrict__ vout, int shift, const unsigned* __restrict__ counts, const SortSeg* __restrict__ sg,
    unsigned n_regions, unsigned miss, unsigned n_bags, const unsigned* __restrict__ tile_reg) {
  extern __shared__ unsigned smem[];
  unsigned(*cnt)[kDigits] = reinterpret_cast<unsigned(*)[kDigits]>(smem);  // [kSortWarps][kDigits]
  unsigned* gbase = smem + kSortWarps * kDigits;                             // [kDigits]
  unsigned* wtot = gbase + kDigits;                                           // [33]
  uint2* tkv = reinterpret_cast<uint2*>(wtot + 34);                          // [kSortTile] (8-byte aligned)
  __shared__ unsigned reg;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned tile = blockIdx.x;
  if (threadIdx.x == 0) reg = tile_reg ? tile_reg[tile] : region_of_tile(sg, n_regions, tile);
  __syncthreads();
  const unsigned r = reg;
  if (r == n_regions) return;  // a spare tile
  const SortSeg g = sg[r];
  const unsigned nt = sg[r + 1].tile0 - g.tile0, lt = tile - g.tile0;
  const unsigned lo = g.lo + lt * kSortTile, hi = min(lo + kSortTile, g.hi);
  for (int i = threadIdx.x; i < kSortWarps * kDigits; i += kSortThreads) smem[i] = 0;
  for (int dg = threadIdx.x; dg < kDigits; dg += kSortThreads)
    gbase[dg] = counts[(size_t)kDigits * g.tile0 + (size_t)dg * nt + lt];
  __syncthreads();
  const unsigned base = lo + w * 32 * kSortItems;
  unsigned k[kSortItems], v[kSortItems], d[kSortItems], rank[kSortItems];
  bool valid[kSortItems];
#pragma unroll
  for (int q = 0; q < kSortItems; ++q) {
    const unsigned i = base + q * 32 + lane;
    valid[q] = i < hi;
    k[q] = valid[q] ? (g.absent ? miss : kin[i]) : 0;
    v[q] = valid[q] ? (g.absent ? n_bags : vin[i]) : 0;
    d[q] = region_digit(g, k[q], shift);
  }
  warp_rank(d, rank, valid, cnt[w]);
  __syncthreads();
  // digit totals of the tile and per-(digit, warp) offsets, digit-major
  static_assert(kDigits % kSortThreads == 0 || kSortThreads % kDigits == 0, "digit/thread split");
  constexpr int kPer = kDigits >= kSortThreads ? kDigits / kSortThreads : 1;
  unsigned run[kPer];
  unsigned mytot = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int dg = threadIdx.x * kPer + j;
    unsigned acc = 0;
    if (dg < kDigits) {
#pragma unroll
      for (int ww = 0; ww < kSortWarps; ++ww) {
        unsigned c = cnt[ww][dg];
        cnt[ww][dg] = acc;
        acc += c;
      }
    }
    run[j] = acc;
    mytot += acc;
  }
  __syncthreads();
  unsigned excl = block_excl_scan(mytot, wtot);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int dg = threadIdx.x * kPer + j;
    if (dg < kDigits) {
      gbase[dg] -= excl;  // now output position minus tile position for the digit
#pragma unroll
      for (int ww = 0; ww < kSortWarps; ++ww) cnt[ww][dg] += excl;
      excl += run[j];
    }
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < kSortItems; ++q) {
    if (valid[q]) {
      const unsigned pos = cnt[w][d[q]] + rank[q];
      tkv[pos] = make_uint2(k[q], v[q]);
    }
  }
  __syncthreads();
  const unsigned tile_n = hi - lo;
  for (unsigned j = threadIdx.x; j < tile_n; j += kSortThreads) {
    const uint2 kv = tkv[j];
    const unsigned kk = kv.x;
    const unsigned dg = region_digit(g, kk, shift);
    const unsigned gp = gbase[dg] + j;
    kout[gp] = kk;
    vout[gp] = kv.y;
  }
}

// ------------------------------------------------------------------ scan (u32, exclusive)

__global__ void __launch_bounds__(kScanThreads) scan_reduce_kernel(const unsigned* __restrict__ in, size_t n,
                                                                   unsigned* __restrict__ partials) {
  __shared__ unsigned wt[33];
  const size_t base = (size_t)blockIdx.x * kScanTile;
  unsigned s = 0;
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    size_t i = base + (size_t)j * kScanThreads + threadIdx.x;
    if (i < n) s += in[i];
  }
  block_excl_scan(s, wt);
  if (threadIdx.x == 0) partials[blockIdx.x] = wt[32];
}

// single block: exclusive scan of the partials in place; total to partials[np]
__global__ void __launch_bounds__(1024) scan_partials_kernel(unsigned* partials, unsigned np) {
  __shared__ unsigned wt[32];
  __shared__ unsigned carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (unsigned b0 = 0; b0 < np; b0 += 1024) {
    const unsigned i = b0 + threadIdx.x;
    const unsigned v = i < np ? partials[i] : 0;
    // block scan with 1024 threads
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    unsigned x = v;
    for (int o = 1; o < 32; o <<= 1) {
      unsigned y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wt[w] = x;
    __syncthreads();
    if (w == 0) {
      unsigned t = wt[lane], incl = t;
      for (int o = 1; o < 32; o <<= 1) {
        unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      wt[lane] = incl - t;
    }
    __syncthreads();
    const unsigned excl = carry + wt[w] + x - v;
    if (i < np) partials[i] = excl;
    __syncthreads();
    if (threadIdx.x == 1023) carry = excl + v;
    __syncthreads();
  }
  if (threadIdx.x == 0) partials[np] = carry;
}

__global__ void __launch_bounds__(kScanThreads) scan_down_kernel(const unsigned* __restrict__ in,
                                                                 unsigned* __restrict__ out, size_t n,
                                                                 const unsigned* __restrict__ partials) {
  __shared__ unsigned wt[33];
  // blocked arrangement: thread t owns kScanItems consecutive elements
  const size_t base = (size_t)blockIdx.x * kScanTile + (size_t)threadIdx.x * kScanItems;
  // a whole run of kScanItems in range moves as 16-byte vectors (in and out
  // are 16-byte aligned and base is a multiple of 16 elements)
  const bool whole = base + kScanItems <= n;
  unsigned v[kScanItems];
  unsigned s = 0;
  if (whole) {
#pragma unroll
    for (int j = 0; j < kScanItems; j += 4) {
      const uint4 x = *reinterpret_cast<const uint4*>(in + base + j);
      v[j] = x.x; v[j + 1] = x.y; v[j + 2] = x.z; v[j + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kScanItems; ++j) v[j] = base + j < n ? in[base + j] : 0;
  }
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) s += v[j];
  unsigned excl = block_excl_scan(s, wt) + partials[blockIdx.x];
  unsigned o[kScanItems];
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    o[j] = excl;
    excl += v[j];
  }
  if (whole) {
#pragma unroll
    for (int j = 0; j < kScanItems; j += 4)
      *reinterpret_cast<uint4*>(out + base + j) = make_uint4(o[j], o[j + 1], o[j + 2], o[j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < kScanItems; ++j)
      if (base + j < n) out[base + j] = o[j];
  }
}

// ------------------------------------------------------------------ placement of the pairs
//
// The pair of every occurrence is written straight into the region of its
// feature slot, in slot-major order: the bags of slot 0 (b ascending), then
// those of slot 1, and so on; within a bag, in key order.  Rows are numbered
// slot-major, so the stable sort then only orders each slot's in-slot row
// numbers: at 64 slots of 1.56M keys 21 bits (3 passes of 7) instead of 27
// (4 passes), and the occurrences of a row keep the order they had before
// (the bags of its slot in b order), so the per-row sums are unchanged.
// dest[t], t = s * B + b, is the exclusive prefix sum of the bag lengths in
// slot-major order, each clamped exactly as the forward clamps malformed
// offsets: the first position of bag b * S + s's pairs.

// Bag lengths (clamped as the forward clamps them) in slot-major order:
// Lt[s * B + b] = length of bag b * S + s.  A 32 x 32 tile of (sample, slot)
// per block, read along slots (consecutive offsets) and written along
// samples through shared memory, so both sides are coalesced; each block
// also adds its exact 64-bit sum of lengths to the header's total (zeroed
// beforehand), which equals nnz exactly when the clamped bags tile [0, nnz).
__global__ void __launch_bounds__(256) len_transpose_kernel(const long long* __restrict__ offsets,
                                                            unsigned long long B, unsigned S, long long nnz,
                                                            unsigned* __restrict__ Lt, WsHeader* hdr) {
  __shared__ unsigned tile[32][33];
  __shared__ unsigned long long wsum[8];
  const unsigned tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8 threads
  const unsigned long long b0 = (unsigned long long)blockIdx.x * 32;
  const unsigned s0 = blockIdx.y * 32;
  unsigned long long sum = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const unsigned long long b = b0 + ty + 8 * r;
    const unsigned s = s0 + tx;
    unsigned len = 0;
    if (b < B && s < S) {
      const unsigned long long bag = b * S + s;
      const long long start = min(max(offsets[bag], 0LL), nnz);
      const long long end = min(max(offsets[bag + 1], start), nnz);
      len = (unsigned)(end - start);
    }
    tile[ty + 8 * r][tx] = len;
    sum += len;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (tx == 0) wsum[ty] = sum;
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const unsigned s = s0 + ty + 8 * r;
    const unsigned long long b = b0 + tx;
    if (b < B && s < S) Lt[(unsigned long long)s * B + b] = tile[tx][ty + 8 * r];
  }
  if (threadIdx.x == 0) {
    unsigned long long t = 0;
    for (int w = 0; w < 8; ++w) t += wsum[w];
    if (t) atomicAdd(&hdr->total, t);
  }
}

// The region of every sort tile, found once per step: the largest region r
// with sg[r].tile0 <= tile, or n_regions for the spare tiles after the last.
__global__ void tile_map_kernel(const SortSeg* __restrict__ sg, unsigned n_regions, unsigned n_tiles,
                                unsigned* __restrict__ tile_reg) {
  for (unsigned t = blockIdx.x * blockDim.x + threadIdx.x; t < n_tiles; t += gridDim.x * blockDim.x)
    tile_reg[t] = region_of_tile(sg, n_regions, t);
}

// One block: the workspace header and the sort regions.  Region s < S holds
// slot s's pairs, [dest[s * B], dest[(s + 1) * B]) (the last slot ends at
// nnz); region S, the absent
// region, is empty.  If the clamped bag lengths do not add up to nnz
// (malformed offsets; flagged) the bags do not tile [0, nnz): then every
// slot region is empty and the absent region covers all of [0, nnz), so the
// first sort pass overwrites every position with an absent pair and the
// backward updates nothing.
__global__ void __launch_bounds__(1024) seg_setup_kernel(TableView t, WsHeader* hdr, unsigned nnz,
                                                         unsigned long long n_bags, unsigned sorted_in_b,
                                                         const unsigned* __restrict__ dest, SortSeg* __restrict__ sg) {
  __shared__ unsigned wt[33];
  __shared__ unsigned carry;
  const unsigned S = (unsigned)t.n_slots;
  const unsigned long long B = n_bags / S;
  const bool placed = B > 0 && hdr->total == (unsigned long long)nnz;
  if (threadIdx.x == 0) {
    hdr->magic = kMagic;
    hdr->nnz = nnz;
    hdr->n_bags = (unsigned)n_bags;
    hdr->sorted_in_b = sorted_in_b;
    hdr->miss_row = t.n_rows;
    hdr->n_unique = 0;
    hdr->placed = placed ? 1u : 0u;
    carry = 0;
    if (!placed && nnz > 0) atomicOr(t.flags, EMB_FLAG_BAD_OFFSETS);
  }
  __syncthreads();
  for (unsigned r0 = 0; r0 <= S; r0 += blockDim.x) {
    const unsigned r = r0 + threadIdx.x;
    SortSeg g{0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    unsigned nt = 0;
    if (r < S) {
      if (placed) {
        g.lo = dest[(unsigned long long)r * B];
        g.hi = r + 1 < S ? dest[(unsigned long long)(r + 1) * B] : nnz;
      }
      const SlotInfo si = t.sinfo[r];
      g.rbase = si.row_base;
      g.cap = si.n_rows;
    } else if (r == S) {
      g.lo = placed ? nnz : 0u;
      g.hi = nnz;
      g.absent = 1;
    }
    if (r <= S) nt = (g.hi - g.lo + kSortTile - 1) / kSortTile;
    const unsigned ex = block_excl_scan(nt, wt);
    g.tile0 = carry + ex;
    if (r <= S) sg[r] = g;
    __syncthreads();
    if (threadIdx.x == 0) carry += wt[32];
    __syncthreads();
  }
  if (threadIdx.x == 0) sg[S + 1].tile0 = carry;  // tile count
}

// ------------------------------------------------------------------ 3. reduce + Adagrad

// Four consecutive weights as float (one 16-byte f32 or 8-byte f16 access).
__device__ __forceinline__ void ldw4(const float* p, float (&v)[4]) {
  const float4 x = *reinterpret_cast<const float4*>(p);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
__device__ __forceinline__ void ldw4(const __half* p, float (&v)[4]) {
  const uint2 x = *reinterpret_cast<const uint2*>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&x.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&x.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
// Updated weights and accumulators are written with streaming (evict-first)
// stores: a row is not touched again in the step, and its lines would
// otherwise push the grad_out columns the reduce keeps reusing out of L2
// (measured 13.9 -> 13.6 ms at 100M keys x dim 128).
__device__ __forceinline__ void stw4(float* p, const float (&v)[4]) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
}
__device__ __forceinline__ void stw4(__half* p, const float (&v)[4]) {
  const __half2 a = __floats2half2_rn(v[0], v[1]);  // round-to-nearest-even
  const __half2 b = __floats2half2_rn(v[2], v[3]);
  uint2 x;
  x.x = *reinterpret_cast<const unsigned*>(&a);
  x.y = *reinterpret_cast<const unsigned*>(&b);
  __stcs(reinterpret_cast<uint2*>(p), x);
}

// ------------------------------------------------------------------ optimizers
//
// The update every element of a hit row receives, given its summed gradient g.

// Adagrad (JD ads article 3.2.1):  acc += g*g;  w -= lr*g / (sqrt(acc) + eps).
// sqrt(acc) is acc * rsqrt(acc) and the quotient a fast divide (hardware
// reciprocal square root and reciprocal, each within a few ulp), which keeps
// the update well inside the float32 tolerance at a fraction of the
// instructions of the correctly rounded sequences.
struct AdagradStep {
  static constexpr bool kZ = false;        // no second state array
  static constexpr bool kRowWise = false;  // one accumulator per element
  float lr, eps;
  __device__ __forceinline__ void elem(float& w, float& a, float& /*z*/, float g) const {
    a = fmaf(g, g, a);
    const float sq = a > 0.f ? a * rsqrtf(a) : 0.f;
    w -= __fdividef(lr * g, sq + eps);
  }
};

// FTRL-Proximal, the other sparse optimizer the JD ads article names (3.2.1),
// in the per-coordinate form of McMahan et al., "Ad Click Prediction: a View
// from the Trenches" (KDD 2013), Algorithm 1; the accumulator array holds n
// and a second array holds z:
//   sigma = (sqrt(n + g*g) - sqrt(n)) / alpha;  z += g - sigma * w;  n += g*g;
//   w = 0 if |z| <= lambda1, else -(z - sign(z) lambda1) / ((beta + sqrt(n)) / alpha + lambda2)
// with w on the right of the z update the weight the forward used.  Correctly
// rounded float32 operations in this order, none contracted: the difference
// of square roots cancels when g*g << n, and the same rounding sequence as
// the oracle's keeps that cancellation identical on both sides.
struct FtrlStep {
  static constexpr bool kZ = true;
  static constexpr bool kRowWise = false;
  float alpha, beta, l1, l2;
  __device__ __forceinline__ void elem(float& w, float& n, float& z, float g) const {
    const float n1 = __fadd_rn(n, __fmul_rn(g, g));
    const float sn = __fsqrt_rn(n), sn1 = __fsqrt_rn(n1);
    const float sigma = __fdiv_rn(__fsub_rn(sn1, sn), alpha);
    z = __fsub_rn(__fadd_rn(z, g), __fmul_rn(sigma, w));
    n = n1;
    if (fabsf(z) <= l1) {
      w = 0.f;
    } else {
      const float num = __fsub_rn(z, z > 0.f ? l1 : -l1);
      const float den = __fadd_rn(__fdiv_rn(__fadd_rn(beta, sn1), alpha), l2);
      w = -__fdiv_rn(num, den);
    }
  }
};

// Row-wise Adagrad: Adagrad with one accumulator per row (key) instead of
// one per element.  The pages give no formula for this variant; the reading
// here adds the mean of the row's squared gradient:  a += (sum_d g_d^2) / D;
// then every element  w -= lr*g / (sqrt(a) + eps), with the same fast sqrt and
// divide as AdagradStep.  The accumulator array holds one f32 per row.
struct RowAdagradStep {
  static constexpr bool kZ = false;
  static constexpr bool kRowWise = true;
  float lr, eps;
};

// The update of 4 consecutive elements from e: weights, accumulators (and z)
// read, updated and written back with evict-first stores; for master-copy
// tables (W the f32 masters) the f16 copy the forward reads is written from
// the new masters too, rounded to nearest-even.
template <typename TW, typename Opt>
__device__ __forceinline__ void update4(const TableView& t, long long e, const float* g, const Opt& o) {
  TW* W = static_cast<TW*>(t.W);
  const float4 a = *reinterpret_cast<const float4*>(t.ACC + e);
  float av[4] = {a.x, a.y, a.z, a.w};
  float zv[4] = {0.f, 0.f, 0.f, 0.f};
  if (Opt::kZ) {
    const float4 z = *reinterpret_cast<const float4*>(t.Z + e);
    zv[0] = z.x; zv[1] = z.y; zv[2] = z.z; zv[3] = z.w;
  }
  float wv[4];
  ldw4(W + e, wv);
#pragma unroll
  for (int j = 0; j < 4; ++j) o.elem(wv[j], av[j], zv[j], g[j]);
  __stcs(reinterpret_cast<float4*>(t.ACC + e), make_float4(av[0], av[1], av[2], av[3]));
  if (Opt::kZ) __stcs(reinterpret_cast<float4*>(t.Z + e), make_float4(zv[0], zv[1], zv[2], zv[3]));
  stw4(W + e, wv);
  if (std::is_same<TW, float>::value && t.W16) stw4(t.W16 + e, wv);
}

// The update on one lane's columns of one row (the fixup).
template <typename TW, int NCB, typename Opt>
__device__ __forceinline__ void update_row(const TableView& t, long long e0, int D, int G, int li,
                                           const float (&g)[NCB][4], const Opt& o) {
#pragma unroll
  for (int c = 0; c < NCB; ++c) {
    const int ce = (c * G + li) * 4;
    if (ce < D) update4<TW>(t, e0 + ce, g[c], o);
  }
}

__device__ __forceinline__ void row_geom(const TableView& t, unsigned row, int& D, int& col, long long& e0) {
  if (t.uniform_dim) {
    D = t.uniform_dim;
    const int s = key_slot(t.row_key[row]);
    col = s * D;
    e0 = (long long)row * D;
  } else {
    const int s = key_slot(t.row_key[row]);
    const SlotInfo si = t.sinfo[s];
    D = si.dim;
    col = si.col;
    e0 = row_elem(si, row);
  }
}

// The update on VW consecutive columns starting at element e (VW a multiple of 4).
template <typename TW, int VW, typename Opt>
__device__ __forceinline__ void update_cols(const TableView& t, long long e, const float* g, const Opt& o) {
#pragma unroll
  for (int h = 0; h < VW; h += 4) update4<TW>(t, e + h, g + h, o);
}

// Row-wise Adagrad on one row whose gradient is spread over a group of G
// lanes: lane li holds columns (cc*G + li)*4 + j, j < 4, in g[cc][j].  The
// squared gradient is summed per lane (columns ascending) and then across
// the group with a fixed xor tree (deterministic); every lane of the group
// computes the new accumulator, lane 0 writes it, and each lane updates its
// own weights (and, for master-copy tables, their f16 copy).
template <typename TW, int G, int NCB>
__device__ __forceinline__ void rowwise_update(const TableView& t, unsigned row, long long e0, int D, int li,
                                               unsigned gmask, const float (&g)[NCB][4], const RowAdagradStep& o) {
  float ss = 0.f;
#pragma unroll
  for (int cc = 0; cc < NCB; ++cc) {
    const int col = (cc * G + li) * 4;
    if (col < D)
#pragma unroll
      for (int j = 0; j < 4; ++j) ss = fmaf(g[cc][j], g[cc][j], ss);
  }
#pragma unroll
  for (int off = 1; off < G; off <<= 1) ss += __shfl_xor_sync(gmask, ss, off, G);
  const float a = t.ACC[row] + ss / (float)D;
  __syncwarp(gmask);  // every lane has read the old accumulator
  if (li == 0) t.ACC[row] = a;
  const float den = (a > 0.f ? a * rsqrtf(a) : 0.f) + o.eps;
  TW* W = static_cast<TW*>(t.W);
#pragma unroll
  for (int cc = 0; cc < NCB; ++cc) {
    const int col = (cc * G + li) * 4;
    if (col < D) {
      float wv[4];
      ldw4(W + e0 + col, wv);
#pragma unroll
      for (int j = 0; j < 4; ++j) wv[j] -= __fdividef(o.lr * g[cc][j], den);
      stw4(W + e0 + col, wv);
      if (std::is_same<TW, float>::value && t.W16) stw4(t.W16 + e0 + col, wv);
    }
  }
}

// Geometry of a row taken from the feature slot of a bag that holds it (the
// expand step only pairs a row with bags of its own slot).  ok is false for a
// row outside that slot's range, which only stale workspace data can produce.
struct RowGeo {
  long long e0;
  int D;
  int col;
  bool ok;
};

__device__ __forceinline__ RowGeo geo_from_slot(const TableView& t, unsigned row, int s) {
  RowGeo g;
  if (t.uniform_dim) {
    g.D = t.uniform_dim;
    g.col = s * g.D;
    g.ok = row < t.n_rows;
    g.e0 = (long long)row * g.D;
  } else {
    const SlotInfo si = t.sinfo[s];
    g.D = si.dim;
    g.col = si.col;
    g.ok = row >= si.row_base && row - si.row_base < si.n_rows;
    g.e0 = g.ok ? row_elem(si, row) : 0;
  }
  return g;
}

__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// The weight and accumulator bytes of a row, pulled towards L2 ahead of its
// read-modify-write.
template <typename TW, bool kRowAcc>
__device__ __forceinline__ void prefetch_row(const TableView& t, const RowGeo& g, unsigned row) {
  const char* w = reinterpret_cast<const char*>(static_cast<const TW*>(t.W) + g.e0);
  for (int o = 0; o < g.D * (int)sizeof(TW); o += 128) prefetch_l2(w + o);
  if (kRowAcc) {
    prefetch_l2(t.ACC + row);
  } else {
    const char* a = reinterpret_cast<const char*>(t.ACC + g.e0);
    for (int o = 0; o < g.D * 4; o += 128) prefetch_l2(a + o);
  }
}

// VW consecutive floats of grad_out: one 16-byte read-only load.
template <int VW>
struct GradVec;
template <>
struct GradVec<4> {
  float v[4];
  __device__ __forceinline__ void load(const float* p) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  }
};

// acc[i] += w * g[i] for an even count, two lanes of fp32 per instruction.
template <int N>
__device__ __forceinline__ void fma_x2(float* acc, float w, const float* g) {
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    unsigned long long a, x, ww, r;
    asm("mov.b64 %0, {%1,%2};" : "=l"(a) : "f"(acc[i]), "f"(acc[i + 1]));
    asm("mov.b64 %0, {%1,%2};" : "=l"(x) : "f"(g[i]), "f"(g[i + 1]));
    asm("mov.b64 %0, {%1,%1};" : "=l"(ww) : "f"(w));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(ww), "l"(x), "l"(a));
    asm("mov.b64 {%0,%1}, %2;" : "=f"(acc[i]), "=f"(acc[i + 1]) : "l"(r));
  }
}

// Knuth's TwoSum on pairs of floats: s + x == t + e exactly with t = fl(s + x);
// s becomes t and the rounding error e is added to the compensation c, so
// s + c carries the running sum to about one rounding of its exact value
// however long the run (a plain float32 running sum loses up to one ulp of
// the running sum per addition).  Packed f32x2 arithmetic in inline PTX, so
// no step is contracted or reassociated.
template <int N>
__device__ __forceinline__ void two_sum_x2(float* s, float* c, const float* x) {
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    unsigned long long S, X, C, T, Z, A, B;
    asm("mov.b64 %0, {%1,%2};" : "=l"(S) : "f"(s[i]), "f"(s[i + 1]));
    asm("mov.b64 %0, {%1,%2};" : "=l"(X) : "f"(x[i]), "f"(x[i + 1]));
    asm("mov.b64 %0, {%1,%2};" : "=l"(C) : "f"(c[i]), "f"(c[i + 1]));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(T) : "l"(S), "l"(X));  // t = s + x
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(Z) : "l"(T), "l"(S));  // z = t - s
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(A) : "l"(T), "l"(Z));  // t - z
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(A) : "l"(S), "l"(A));  // s - (t - z)
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(B) : "l"(X), "l"(Z));  // x - z
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(A) : "l"(A), "l"(B));  // e
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(C) : "l"(C), "l"(A));  // c += e
    asm("mov.b64 {%0,%1}, %2;" : "=f"(s[i]), "=f"(s[i + 1]) : "l"(T));
    asm("mov.b64 {%0,%1}, %2;" : "=f"(c[i]), "=f"(c[i + 1]) : "l"(C));
  }
}

// The same TwoSum step on one float.
__device__ __forceinline__ void two_sum(float& s, float& c, float x) {
  const float t = __fadd_rn(s, x);
  const float z = __fsub_rn(t, s);
  c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, __fsub_rn(t, z)), __fsub_rn(x, z)));
  s = t;
}

struct StageMeta {
  long long e0;
  unsigned row;
  int D;
  int flags;  // bit0: segment starts in this sub-chunk, bit1: ends in it
};

// One lane group of G lanes streams a sub-chunk of `chunk` sorted positions;
// each lane owns VW-float column vectors (NCB of them) of the row.  Per
// window of G positions the lanes first work in parallel, one position each:
// row, bag, merged run of equal (row, bag) neighbours, its weight (1/L times
// the run length), the address of its grad_out columns, and whether a new
// row starts there; each lane leaves that as a 16-byte record in shared
// memory, and lanes that start a row prefetch its weights and accumulators
// into L2.  The group then walks the window in order, U positions at a time:
// per position one broadcast read of the record and one vector load per
// column block, then multiply-adds; a group of U positions with no row start
// in it adds without any per-position test.  The U products of a group are
// summed plainly and the group's sum is folded into the row's running sum
// with TwoSum (a compensated float32 sum: about one rounding of the exact
// per-key gradient however many occurrences a hot key has).  At a row start
// the finished row is staged in shared memory.  Staged rows are then applied (Adagrad on a
// whole segment) or parked (partial of a segment cut by a sub-chunk edge) by
// one copy of that code, outside the unrolled walk.
constexpr int kRedWarps = 4;  // warps per reduce block

struct alignas(16) PosRec {
  const float* p;  // the position's grad_out columns, or the zero row for a position that adds nothing
  float w;         // its weight: (1/L or 1) x the run of equal (row, bag) positions it stands for, or 0
  int D;           // dim of its slot (columns at or past it read the zero row)
};

// acc[i] += w * g[i] for VW columns.
template <int VW>
__device__ __forceinline__ void fma_vw(float* acc, float w, const float* g) {
  fma_x2<VW>(acc, w, g);
}

// kAllCols: every lane column is inside every row (one dim, equal to G x VW x NCB).
template <typename TW, int G, int VW, int NCB, int U, bool kAllCols, typename Opt>
__global__ void __launch_bounds__(kRedWarps * 32, 8) segreduce_update_kernel(
    TableView t, const unsigned* __restrict__ K, const unsigned* __restrict__ V, const float* __restrict__ scale,
    int mean, const float* __restrict__ grad, const float* __restrict__ zrow, unsigned n, unsigned n_bags,
    unsigned n_chunks, unsigned chunk, float* __restrict__ partA, float* __restrict__ partB,
    unsigned* __restrict__ arow, Opt opt,
    unsigned* __restrict__ work) {
  constexpr int P = 32 / G;
  constexpr int CW = G * VW * NCB;      // columns a group covers
  constexpr int UW = U < G ? U : G;     // positions per walk step (a window holds G)
  constexpr int kStage = UW + 1;
  __shared__ __align__(16) float stage[kRedWarps][P][kStage][CW];
  __shared__ StageMeta meta[kRedWarps][P][kStage];
  __shared__ PosRec recs[kRedWarps][P][G];
  __shared__ uint2 srecs[kRedWarps][P][G];  // (row, bag) of each walked row start
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int sub = lane / G, li = lane % G;
  const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (sub * G));
  const unsigned gbits = G == 32 ? 0xffffffffu : ((1u << G) - 1u);
  const unsigned S = (unsigned)t.n_slots;
  const unsigned miss = t.n_rows;
  const int maxd = t.max_dim;
  const int udim = t.uniform_dim;
  float(*st)[CW] = stage[wid][sub];
  StageMeta* mt = meta[wid][sub];
  PosRec* rc = recs[wid][sub];
  uint2* sr = srecs[wid][sub];
  const unsigned n_groups = ((gridDim.x * blockDim.x) >> 5) * P;
  // sub-chunks: a static grid-stride order, or (work != NULL) taken in order from a counter
  auto next_chunk = [&](unsigned c) -> unsigned {
    if (!work) return c + n_groups;
    unsigned v = 0;
    if (li == 0) v = atomicAdd(work, 1u);
    return __shfl_sync(gmask, v, 0, G);
  };
  const unsigned c_first = work ? next_chunk(0) : ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * P + sub;
  for (unsigned c = c_first; c < n_chunks; c = next_chunk(c)) {
    const unsigned cs = c * chunk;
    const unsigned ce = min(cs + chunk, n);
    const unsigned before = cs > 0 ? K[cs - 1] : kNoRow;
    const bool first_starts = K[cs] != before;
    const bool last_ends = ce >= n || K[ce] != K[ce - 1];
    if (li == 0) arow[c] = kNoRow;
    unsigned cur = kNoRow;
    bool cur_starts = first_starts;
    RowGeo cg{0, 0, 0, false};
    float acc[NCB][VW];  // running sum of the row
    float cmp[NCB][VW];  // its TwoSum compensation
#pragma unroll
    for (int cc = 0; cc < NCB; ++cc)
#pragma unroll
      for (int j = 0; j < VW; ++j) acc[cc][j] = cmp[cc][j] = 0.f;

    // stage the finished row `cur` (no-op for misses and stale rows)
    auto stage_cur = [&](int slot, bool ends) {
#pragma unroll
      for (int cc = 0; cc < NCB; ++cc)
#pragma unroll
        for (int j = 0; j < VW; j += 4)
          *reinterpret_cast<float4*>(&st[slot][(cc * G + li) * VW + j]) =
              make_float4(__fadd_rn(acc[cc][j], cmp[cc][j]), __fadd_rn(acc[cc][j + 1], cmp[cc][j + 1]),
                          __fadd_rn(acc[cc][j + 2], cmp[cc][j + 2]), __fadd_rn(acc[cc][j + 3], cmp[cc][j + 3]));
      if (li == 0) mt[slot] = StageMeta{cg.e0, cur, (cur < miss && cg.ok) ? cg.D : 0,
                                        (cur_starts ? 1 : 0) | (ends ? 2 : 0)};
    };
    // apply or park the staged rows [0, ns)
    auto drain = [&](int ns) {
      __syncwarp(gmask);
      for (int f = 0; f < ns; ++f) {
        const StageMeta sm = mt[f];
        if (sm.D == 0) continue;
        if (sm.flags == 3) {
          if constexpr (Opt::kRowWise) {
            static_assert(VW == 4, "row-wise update takes 4 columns per lane block");
            float gr[NCB][4];
#pragma unroll
            for (int cc = 0; cc < NCB; ++cc) {
              const int col = (cc * G + li) * VW;
#pragma unroll
              for (int j = 0; j < 4; ++j) gr[cc][j] = col < sm.D ? st[f][col + j] : 0.f;
            }
            rowwise_update<TW, G, NCB>(t, sm.row, sm.e0, sm.D, li, gmask, gr, opt);
          } else {
#pragma unroll
            for (int cc = 0; cc < NCB; ++cc) {
              const int col = (cc * G + li) * VW;
              if (col < sm.D) update_cols<TW, VW>(t, sm.e0 + col, &st[f][col], opt);
            }
          }
        } else {
          float* dst = ((sm.flags & 1) ? partA : partB) + (size_t)c * maxd;
          if ((sm.flags & 1) && li == 0) arow[c] = sm.row;
#pragma unroll
          for (int cc = 0; cc < NCB; ++cc) {
            const int col = (cc * G + li) * VW;
            if (col < sm.D) {
#pragma unroll
              for (int j = 0; j < VW; j += 4)
                *reinterpret_cast<float4*>(dst + col + j) = *reinterpret_cast<const float4*>(&st[f][col + j]);
            }
          }
        }
      }
      __syncwarp(gmask);
    };

    unsigned prev_row = before;
    // One-dim tables load each window's (row, bag) pairs while the previous
    // window is walked (measured: 14.34 ms against 14.71 at 100M keys); on
    // ragged tables the two extra registers spill and it loses (0.683 ms
    // against 0.660), so they load at the window's start.
    unsigned kk_n = 0, vv_n = 0;
    if (kAllCols) {
      kk_n = cs + li < ce ? K[cs + li] : kNoRow;
      vv_n = cs + li < ce ? V[cs + li] : 0u;
    }
    for (unsigned i0 = cs; i0 < ce; i0 += G) {
      // ---- lane-parallel bookkeeping, one position per lane
      const int m = (int)min((unsigned)G, ce - i0);
      const bool valid = li < m;
      unsigned kk, vv;
      if (kAllCols) {
        kk = kk_n;
        vv = vv_n;
        const bool nx = i0 + G + li < ce;
        kk_n = nx ? K[i0 + G + li] : kNoRow;
        vv_n = nx ? V[i0 + G + li] : 0u;
      } else {
        kk = valid ? K[i0 + li] : kNoRow;
        vv = valid ? V[i0 + li] : 0u;
      }
      unsigned kp = __shfl_up_sync(gmask, kk, 1, G);
      const unsigned vp = __shfl_up_sync(gmask, vv, 1, G);
      if (li == 0) kp = prev_row;
      prev_row = __shfl_sync(gmask, kk, m - 1, G);
      const bool dup = valid && li > 0 && kk == kp && vv == vp;
      const unsigned dm = (__ballot_sync(gmask, dup) >> (sub * G)) & gbits;
      const unsigned above = li + 1 < 32 ? (~dm) & ~((2u << li) - 1u) : 0u;
      const int nxt = min(above ? __ffs(above) - 1 : G, m);
      const bool use = valid && !dup && kk < miss && vv < n_bags;
      const bool start = valid && (kk != kp || (i0 == cs && li == 0));
      // Only positions that add something or start a row are walked: merged
      // duplicates, and misses after the first position of their run, are
      // dropped (30% of the positions with Zipf bag lengths up to 256).  The
      // kept ones take consecutive walk indices in window order; smask marks
      // the walk indices of row starts.  The sub-chunk's first position is a
      // start, so it is walk index 0 of the sub-chunk's first window.
      const bool keep = use || start;
      const unsigned kmask = (__ballot_sync(gmask, keep) >> (sub * G)) & gbits;
      const int nk = __popc(kmask);
      const int rank = __popc(kmask & ((1u << li) - 1u));
      unsigned smask = 0;
      for (unsigned sw = (__ballot_sync(gmask, start) >> (sub * G)) & gbits; sw; sw &= sw - 1u)
        smask |= 1u << __popc(kmask & ((1u << (__ffs(sw) - 1)) - 1u));
      const int nw = (nk + UW - 1) / UW * UW;  // walk length, whole steps of UW
      int sj = 0;
      {
        PosRec r{zrow, 0.f, CW};
        if (use) {
          if (udim) {
            r.p = grad + (size_t)vv * (unsigned)udim;   // (b*S + s) * D = b * sum_dims + s * D
            r.D = udim;
          } else {
            sj = (int)(vv % S);
            const SlotInfo si = t.sinfo[sj];
            r.p = grad + (size_t)(vv / S) * (unsigned)t.sum_dims + (unsigned)si.col;
            r.D = si.dim;
          }
          r.w = (mean ? scale[vv] : 1.f) * (float)(nxt - li);
        }
        if (keep) rc[rank] = r;
        if (li >= nk && li < nw) rc[li] = PosRec{zrow, 0.f, CW};  // dead tail of the last step
        if (start) sr[rank] = make_uint2(kk, vv);
      }
      if (use && start) {
        const RowGeo g = geo_from_slot(t, kk, sj);
        if (g.ok) prefetch_row<TW, Opt::kRowWise>(t, g, kk);
      }
      __syncwarp(gmask);
      // ---- in-order walk of the kept positions, U in flight per lane.  Walk
      // indices past the kept ones hold dead records (zero row, weight 0), so
      // every step takes UW positions without bound tests.
#pragma unroll 1  // unrolling the window overflows the instruction cache (measured 2.4x slower)
      for (int j0 = 0; j0 < nw; j0 += UW) {
        GradVec<VW> gv[UW][NCB];
        float wv[UW];
#pragma unroll
        for (int u = 0; u < UW; ++u) {
          const PosRec r = rc[j0 + u];
          wv[u] = r.w;
#pragma unroll
          for (int cc = 0; cc < NCB; ++cc) {
            const int q = (cc * G + li) * VW;
            gv[u][cc].load((kAllCols || q < r.D) ? r.p + q : zrow + q);
          }
        }
        const unsigned grp = (smask >> j0) & ((1u << UW) - 1u);
        if (grp == 0) {
          float blk[NCB][VW];  // plain sum of the group's products
#pragma unroll
          for (int cc = 0; cc < NCB; ++cc)
#pragma unroll
            for (int q = 0; q < VW; ++q) blk[cc][q] = 0.f;
#pragma unroll
          for (int u = 0; u < UW; ++u)
#pragma unroll
            for (int cc = 0; cc < NCB; ++cc) fma_vw<VW>(blk[cc], wv[u], gv[u][cc].v);
#pragma unroll
          for (int cc = 0; cc < NCB; ++cc) two_sum_x2<VW>(acc[cc], cmp[cc], blk[cc]);
        } else {
          // a row starts in this group: every product is folded in on its own
          int ns = 0;
#pragma unroll
          for (int u = 0; u < UW; ++u) {
            const int j = j0 + u;
            if ((grp >> u) & 1u) {
              if (cur != kNoRow) stage_cur(ns++, true);
              const uint2 sv = sr[j];
              cur = sv.x;
              const unsigned bag = sv.y;
              // walk index 0 of the sub-chunk's first window is its first position
              cur_starts = i0 > cs || j > 0 || first_starts;
              cg = (cur < miss && bag < n_bags) ? geo_from_slot(t, cur, (int)(bag % S)) : RowGeo{0, 0, 0, false};
#pragma unroll
              for (int cc = 0; cc < NCB; ++cc)
#pragma unroll
                for (int q = 0; q < VW; ++q) acc[cc][q] = cmp[cc][q] = 0.f;
            }
#pragma unroll
            for (int cc = 0; cc < NCB; ++cc) {
              float p[VW];
#pragma unroll
              for (int q = 0; q < VW; ++q) p[q] = 0.f;
              fma_vw<VW>(p, wv[u], gv[u][cc].v);
              two_sum_x2<VW>(acc[cc], cmp[cc], p);
            }
          }
          if (ns) drain(ns);
        }
      }
      __syncwarp(gmask);  // the next window rewrites the records
    }
    if (cur != kNoRow) {
      stage_cur(0, last_ends);
      drain(1);
    }
  }
}

// ------------------------------------------------------------------ 4. fixup of spanning segments

// Partial-row loads in flight per lane: 8 measured 0.64 ms at 100M keys,
// against 0.75 with 4 and 0.85 with 16.
constexpr int kFixupLoads = 8;

// Folds the partial rows of every block of kFoldChunks sub-chunks that lies
// inside one row's run (the row began before the block and lasts through its
// last position, so each of its sub-chunks left one partial of that row) into
// one partial, summed in sub-chunk order by consecutive ranges per lane group
// and a fixed xor tree; every other block is marked unfolded.  A row of
// Zipf-head popularity spans thousands of sub-chunks: the fixup then adds
// about 1/kFoldChunks as many partials for it.
template <int G, int NCB>
__global__ void __launch_bounds__(256) fold_kernel(TableView t, const unsigned* __restrict__ K, unsigned n,
                                                   unsigned n_chunks, unsigned chunk, unsigned n_fold,
                                                   const float* __restrict__ partB, float* __restrict__ partC,
                                                   unsigned* __restrict__ folded) {
  constexpr int P = 32 / G;
  const int lane = threadIdx.x & 31;
  const int sub = lane / G, li = lane % G;
  const int maxd = t.max_dim;
  const unsigned nwarps = (gridDim.x * blockDim.x) >> 5;
  for (unsigned b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < n_fold; b += nwarps) {
    const unsigned c0 = b * kFoldChunks;
    bool fold = false;
    unsigned row = 0;
    if (c0 > 0 && c0 + kFoldChunks <= n_chunks) {
      const size_t p0 = (size_t)c0 * chunk;
      const size_t pe = (size_t)(c0 + kFoldChunks) * chunk;
      const size_t p1 = (pe < (size_t)n ? pe : (size_t)n) - 1;
      row = K[p0];
      fold = row < t.n_rows && K[p0 - 1] == row && K[p1] == row;
    }
    if (lane == 0) folded[b] = fold ? 1u : 0u;
    if (!fold) continue;
    int D, col;
    long long e0;
    row_geom(t, row, D, col, e0);
    constexpr unsigned per = (kFoldChunks + P - 1) / P;
    const unsigned j0 = sub * per, j1 = min(kFoldChunks, j0 + per);
    float acc[NCB][4], cmp[NCB][4];
#pragma unroll
    for (int cc = 0; cc < NCB; ++cc)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[cc][j] = cmp[cc][j] = 0.f;
    constexpr int FB = kFixupLoads / NCB > 0 ? kFixupLoads / NCB : 1;
    for (unsigned jb = j0; jb < j1; jb += FB) {
      float4 x[FB][NCB];
#pragma unroll
      for (int q = 0; q < FB; ++q) {
        const float* src = partB + (size_t)(c0 + jb + q) * maxd;
#pragma unroll
        for (int cc = 0; cc < NCB; ++cc) {
          const int cidx = (cc * G + li) * 4;
          x[q][cc] = (jb + q < j1 && cidx < D) ? *reinterpret_cast<const float4*>(src + cidx)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int q = 0; q < FB; ++q) {
        if (jb + q < j1) {
#pragma unroll
          for (int cc = 0; cc < NCB; ++cc) {
            two_sum(acc[cc][0], cmp[cc][0], x[q][cc].x);
            two_sum(acc[cc][1], cmp[cc][1], x[q][cc].y);
            two_sum(acc[cc][2], cmp[cc][2], x[q][cc].z);
            two_sum(acc[cc][3], cmp[cc][3], x[q][cc].w);
          }
        }
      }
    }
#pragma unroll
    for (int cc = 0; cc < NCB; ++cc)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        for (int off = G; off < 32; off <<= 1) {
          const float so = __shfl_xor_sync(0xffffffffu, acc[cc][j], off);
          const float co = __shfl_xor_sync(0xffffffffu, cmp[cc][j], off);
          two_sum(acc[cc][j], cmp[cc][j], so);
          cmp[cc][j] = __fadd_rn(cmp[cc][j], co);
        }
        acc[cc][j] = __fadd_rn(acc[cc][j], cmp[cc][j]);
      }
    if (sub == 0) {
      float* dst = partC + (size_t)b * maxd;
#pragma unroll
      for (int cc = 0; cc < NCB; ++cc) {
        const int cidx = (cc * G + li) * 4;
        if (cidx < D)
          *reinterpret_cast<float4*>(dst + cidx) = make_float4(acc[cc][0], acc[cc][1], acc[cc][2], acc[cc][3]);
      }
    }
  }
}

template <typename TW, int G, int NCB, typename Opt>
__global__ void __launch_bounds__(256) fixup_kernel(TableView t, const unsigned* __restrict__ K, unsigned n,
                                                    unsigned n_chunks, unsigned chunk,
                                                    const float* __restrict__ partA,
                                                    const float* __restrict__ partB,
                                                    const float* __restrict__ partC,
                                                    const unsigned* __restrict__ folded,  // NULL: none folded
                                                    const unsigned* __restrict__ arow, Opt opt) {
  constexpr int P = 32 / G;
  const int lane = threadIdx.x & 31;
  const int sub = lane / G, li = lane % G;
  const int maxd = t.max_dim;
  const unsigned nwarps = (gridDim.x * blockDim.x) >> 5;
  for (unsigned c = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; c < n_chunks; c += nwarps) {
    const unsigned row = arow[c];
    if (row >= t.n_rows || c + 1 >= n_chunks) continue;
    // last chunk whose first position still holds this row (K is sorted; the
    // row continues into chunk c + 1 because chunk c left a head partial).
    // Exponential search from c + 1: most such rows end in the next chunk.
    unsigned lo = c + 1, step = 1, probe_c = c + 2;
    while (probe_c < n_chunks && K[(size_t)probe_c * chunk] == row) {
      lo = probe_c;
      step <<= 1;
      probe_c = lo + step;
    }
    unsigned hi = min(probe_c, n_chunks) - 1;  // K[lo * chunk] == row, answer in [lo, hi]
    while (lo < hi) {
      const unsigned mid = lo + (hi - lo + 1) / 2;
      if (K[(size_t)mid * chunk] == row) lo = mid; else hi = mid - 1;
    }
    const unsigned c1 = lo;  // partials: A[c], B[c+1..c1]
    int D, col;
    long long e0;
    row_geom(t, row, D, col, e0);
    // the P lane groups take consecutive ranges of the sub-chunks after the
    // head, [c + 1, c1]; group 0 also takes the head partial.  Inside a
    // group's range, a block of kFoldChunks sub-chunks that lies wholly in it
    // and was folded contributes its one folded partial.
    const unsigned span = c1 - c;
    const unsigned per = (span + P - 1) / P;
    const unsigned ga = min(c + 1 + sub * per, c1 + 1), gb = min(ga + per, c1 + 1);  // the group's [ga, gb)
    float acc[NCB][4], cmp[NCB][4];  // compensated (TwoSum) sums of the partial rows
#pragma unroll
    for (int cc = 0; cc < NCB; ++cc)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[cc][j] = cmp[cc][j] = 0.f;
    // partial rows are read kFixupLoads / NCB at a time (loads in flight per
    // lane), then added in order
    constexpr int FB = kFixupLoads / NCB > 0 ? kFixupLoads / NCB : 1;
    bool head = sub == 0;
    unsigned cp = ga;
    while (head || cp < gb) {
      float4 x[FB][NCB];
      unsigned have = 0;
#pragma unroll
      for (int q = 0; q < FB; ++q) {
        const float* src = nullptr;
        if (head) {
          src = partA + (size_t)c * maxd;
          head = false;
        } else if (cp < gb) {
          if (folded && cp % kFoldChunks == 0 && cp + kFoldChunks <= gb && folded[cp / kFoldChunks]) {
            src = partC + (size_t)(cp / kFoldChunks) * maxd;
            cp += kFoldChunks;
          } else {
            src = partB + (size_t)cp * maxd;
            ++cp;
          }
        }
        if (src) have |= 1u << q;
#pragma unroll
        for (int cc = 0; cc < NCB; ++cc) {
          const int cidx = (cc * G + li) * 4;
          x[q][cc] = (src && cidx < D) ? *reinterpret_cast<const float4*>(src + cidx)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int q = 0; q < FB; ++q) {
        if ((have >> q) & 1u) {
#pragma unroll
          for (int cc = 0; cc < NCB; ++cc) {
            two_sum(acc[cc][0], cmp[cc][0], x[q][cc].x);
            two_sum(acc[cc][1], cmp[cc][1], x[q][cc].y);
            two_sum(acc[cc][2], cmp[cc][2], x[q][cc].z);
            two_sum(acc[cc][3], cmp[cc][3], x[q][cc].w);
          }
        }
      }
    }
    // groups hold consecutive ranges: combine (sum, compensation) pairs with a
    // fixed xor tree, then round each to one float
#pragma unroll
    for (int cc = 0; cc < NCB; ++cc)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        for (int off = G; off < 32; off <<= 1) {
          const float so = __shfl_xor_sync(0xffffffffu, acc[cc][j], off);
          const float co = __shfl_xor_sync(0xffffffffu, cmp[cc][j], off);
          two_sum(acc[cc][j], cmp[cc][j], so);
          cmp[cc][j] = __fadd_rn(cmp[cc][j], co);
        }
        acc[cc][j] = __fadd_rn(acc[cc][j], cmp[cc][j]);
      }
    if constexpr (Opt::kRowWise) {
      // after the xor tree every group holds the row's totals; group 0 applies the update
      const unsigned gm = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (sub * G));
      if (sub == 0) rowwise_update<TW, G, NCB>(t, row, e0, D, li, gm, acc, opt);
    } else {
      if (sub == 0) update_row<TW, NCB>(t, e0, D, G, li, acc, opt);
    }
  }
}

// ------------------------------------------------------------------ unique-key export

__global__ void __launch_bounds__(kScanThreads) head_count_kernel(const unsigned* __restrict__ K, size_t n,
                                                                  unsigned miss, unsigned* __restrict__ partials) {
  __shared__ unsigned wt[33];
  const size_t base = (size_t)blockIdx.x * kScanTile + (size_t)threadIdx.x * kScanItems;
  unsigned s = 0;
  for (int j = 0; j < kScanItems; ++j) {
    const size_t i = base + j;
    if (i < n && K[i] < miss && (i == 0 || K[i - 1] != K[i])) ++s;
  }
  block_excl_scan(s, wt);
  if (threadIdx.x == 0) partials[blockIdx.x] = wt[32];
}

__global__ void __launch_bounds__(kScanThreads) head_write_kernel(const unsigned* __restrict__ K, size_t n,
                                                                  unsigned miss, const unsigned* __restrict__ partials,
                                                                  const long long* __restrict__ row_key,
                                                                  long long* __restrict__ keys_out) {
  __shared__ unsigned wt[33];
  const size_t base = (size_t)blockIdx.x * kScanTile + (size_t)threadIdx.x * kScanItems;
  unsigned s = 0;
  for (int j = 0; j < kScanItems; ++j) {
    const size_t i = base + j;
    if (i < n && K[i] < miss && (i == 0 || K[i - 1] != K[i])) ++s;
  }
  unsigned idx = block_excl_scan(s, wt) + partials[blockIdx.x];
  for (int j = 0; j < kScanItems; ++j) {
    const size_t i = base + j;
    if (i < n && K[i] < miss && (i == 0 || K[i - 1] != K[i])) keys_out[idx++] = row_key[K[i]];
  }
}

__global__ void store_count_kernel(const unsigned* partials, unsigned np, long long* out, WsHeader* hdr) {
  *out = partials[np];
  hdr->n_unique = partials[np];
}

// ------------------------------------------------------------------ host side

static int resident_blocks(int threads) { return sm_count() * (2048 / threads); }

static cudaError_t launch_scan(const unsigned* in, unsigned* out, size_t n, unsigned* partials, cudaStream_t st) {
  const unsigned np = (unsigned)((n + kScanTile - 1) / kScanTile);
  scan_reduce_kernel<<<np, kScanThreads, 0, st>>>(in, n, partials);
  scan_partials_kernel<<<1, 1024, 0, st>>>(partials, np);
  scan_down_kernel<<<np, kScanThreads, 0, st>>>(in, out, n, partials);
  return cudaGetLastError();
}

cudaError_t launch_scan_u32(const unsigned* in, unsigned* out, size_t n, unsigned* partials, cudaStream_t st) {
  return launch_scan(in, out, n, partials, st);
}

static size_t scatter_smem() {
  return sizeof(unsigned) * ((size_t)kSortWarps * kDigits + kDigits + 34 + 2 * (size_t)kSortTile);
}

// Record the caller's timing event for a finished backward phase, if any.
static void mark_phase(const emb_table* t, int phase, cudaStream_t st) {
  if (phase < t->n_phase_events && t->phase_events[phase])
    cudaEventRecord((cudaEvent_t)t->phase_events[phase], st);
}

template <typename TW, int G, int VW, int NCB, typename Opt>
static cudaError_t launch_reduce(const emb_table* t, const unsigned* K, const unsigned* V, const float* scale,
                                 int mean, const float* grad, unsigned n, unsigned n_bags, const WsLayout& L, char* ws,
                                 const Opt& opt, cudaStream_t st) {
  constexpr int U = NCB >= 4 ? 1 : 4 / NCB;  // grad_out vectors in flight per lane (measured best at 4)
  constexpr int P = 32 / G;
  TableView v = t->view();
  const int threads = kRedWarps * 32;
  int per_sm = 0;
  const bool all_cols = t->uniform_dim == G * VW * NCB;
  auto kern = all_cols ? segreduce_update_kernel<TW, G, VW, NCB, U, true, Opt>
                       : segreduce_update_kernel<TW, G, VW, NCB, U, false, Opt>;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0);
  long long blocks = ((long long)L.n_chunks + (threads / 32) * P - 1) / ((threads / 32) * P);
  blocks = std::min<long long>(blocks, (long long)std::max(1, per_sm) * sm_count());
  float* pa = (float*)(ws + L.partA);
  float* pb = (float*)(ws + L.partB);
  unsigned* ar = (unsigned*)(ws + L.arow);
  float* zrow = (float*)(ws + L.zero);
  cudaError_t e = cudaMemsetAsync(zrow, 0, (size_t)EMB_MAX_DIM * 4, st);
  if (e != cudaSuccess) return e;
  // sub-chunks are handed out in order from a counter: all resident groups
  // then work inside a narrow window of one feature slot, whose grad_out
  // columns stay in L2 (measured 23.3 -> 17.2 ms against a static grid-stride
  // order at 100M keys x dim 128)
  unsigned* work = (unsigned*)(ws + L.work);
  e = cudaMemsetAsync(work, 0, sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  kern<<<(int)std::max(1LL, blocks), threads, 0, st>>>(
      v, K, V, scale, mean, grad, zrow, n, n_bags, L.n_chunks, L.chunk, pa, pb, ar, opt, work);
  mark_phase(t, 2, st);
  // the fixup reads partial rows four columns per lane
  constexpr int G4 = G * VW / 4 > 32 ? 32 : G * VW / 4;
  constexpr int NCB4 = (G * VW * NCB) / (4 * G4);
  // Rows that span whole blocks of kFoldChunks sub-chunks have those blocks
  // folded first, so the fixup adds one partial per block (measured: fixup
  // 0.63 -> 0.38 ms at 282M positions).  Below 2^24 positions no row is that
  // long and the extra launch only costs time (0.005 ms at 4.5M to 6.5M).
  float* pc = (float*)(ws + L.partC);
  unsigned* fl = nullptr;
  if ((size_t)n >= kFoldFrom) {
    fl = (unsigned*)(ws + L.folded);
    long long kblocks = std::min<long long>(((long long)L.n_fold * 32 + 255) / 256, resident_blocks(256));
    fold_kernel<G4, NCB4><<<(int)std::max(1LL, kblocks), 256, 0, st>>>(v, K, n, L.n_chunks, L.chunk, L.n_fold, pb,
                                                                       pc, fl);
  }
  long long fblocks = std::min<long long>(((long long)L.n_chunks * 32 + 255) / 256, resident_blocks(256));
  fixup_kernel<TW, G4, NCB4, Opt><<<(int)std::max(1LL, fblocks), 256, 0, st>>>(v, K, n, L.n_chunks, L.chunk, pa,
                                                                                   pb, pc, fl, ar, opt);
  mark_phase(t, 3, st);
  return cudaGetLastError();
}

// Lanes per row: one 16-byte vector of grad_out per lane, up to 32 lanes;
// wider rows give each lane several column blocks.  (32-byte vectors with
// half the lanes per row measured slower at 100M keys x dim 128: they cost
// registers, and resident warps matter more here than load width.)
template <typename TW, typename Opt>
static cudaError_t dispatch_reduce(const emb_table* t, const unsigned* K, const unsigned* V, const float* scale,
                                   int mean, const float* grad, unsigned n, unsigned n_bags, const WsLayout& L,
                                   char* ws, const Opt& opt, cudaStream_t st) {
  const int md = t->st.max_dim;
#define EMB_RED(G, VW, NCB) return launch_reduce<TW, G, VW, NCB>(t, K, V, scale, mean, grad, n, n_bags, L, ws, opt, st)
  if (md <= 4) EMB_RED(1, 4, 1);
  if (md <= 8) EMB_RED(2, 4, 1);
  if (md <= 16) EMB_RED(4, 4, 1);
  if (md <= 32) EMB_RED(8, 4, 1);
  if (md <= 64) EMB_RED(16, 4, 1);
  if (md <= 128) EMB_RED(32, 4, 1);
  if (md <= 256) EMB_RED(32, 4, 2);
  EMB_RED(32, 4, 4);
#undef EMB_RED
}

// ------------------------------------------------------------------ stable pair sort for the device table build
//
// The same radix kernels over one region [0, n) with no clamping: sorts the
// pairs (key, value) by the low `bits` bits of key, stably.  Scratch layout:
// two region entries + digit counts + scan partials.

static size_t pair_sort_counts(unsigned n) { return (size_t)kDigits * ((n + kSortTile - 1) / kSortTile + 2); }

size_t pair_sort_scratch_bytes(unsigned n) {
  const size_t nc = pair_sort_counts(n);
  const size_t np = (nc + kScanTile - 1) / kScanTile + 1;
  return align_up(3 * sizeof(SortSeg)) + align_up(nc * 4) + align_up(np * 4);
}

__global__ void pair_region_kernel(SortSeg* sg, unsigned n) {
  const unsigned nt = (n + kSortTile - 1) / kSortTile;
  sg[0] = SortSeg{0u, n, 0u, 0u, 0xFFFFFFFFu, 0u, 0u, 0u};
  sg[1] = SortSeg{n, n, nt, 0u, 0u, 1u, 0u, 0u};
  sg[2] = SortSeg{0u, 0u, nt, 0u, 0u, 0u, 0u, 0u};
}

// Sorted pairs end in (kA, vA) if the pass count is even, else (kB, vB); *in_b says which.
cudaError_t pair_sort(unsigned* kA, unsigned* vA, unsigned* kB, unsigned* vB, unsigned n, int bits, void* scratch,
                      cudaStream_t st, bool* in_b) {
  *in_b = false;
  if (n == 0) return cudaSuccess;
  char* sc = (char*)scratch;
  SortSeg* sg = (SortSeg*)sc;
  const size_t nc = pair_sort_counts(n);
  unsigned* counts = (unsigned*)(sc + align_up(3 * sizeof(SortSeg)));
  unsigned* partials = (unsigned*)(sc + align_up(3 * sizeof(SortSeg)) + align_up(nc * 4));
  const unsigned n_tiles = (unsigned)(nc / kDigits);
  pair_region_kernel<<<1, 1, 0, st>>>(sg, n);
  const size_t smem = scatter_smem();
  cudaError_t e = cudaFuncSetAttribute(radix_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int passes = std::max(1, (bits + kRadixBits - 1) / kRadixBits);
  unsigned *ki = kA, *vi = vA, *ko = kB, *vo = vB;
  for (int p = 0; p < passes; ++p) {
    radix_count_kernel<<<n_tiles, kSortThreads, 0, st>>>(ki, sg, 1u, p * kRadixBits, counts, nullptr);
    if ((e = launch_scan(counts, counts, nc, partials, st)) != cudaSuccess) return e;
    radix_scatter_kernel<<<n_tiles, kSortThreads, smem, st>>>(ki, vi, ko, vo, p * kRadixBits, counts, sg, 1u, 0u, 0u,
                                                             nullptr);
    std::swap(ki, ko);
    std::swap(vi, vo);
  }
  *in_b = (passes & 1) != 0;
  return cudaGetLastError();
}

static int bits_for(unsigned x) {
  int b = 0;
  while (b < 32 && (x >> b) != 0) ++b;
  return b;
}

// Radix passes: in-slot row numbers and the miss code (the slot's row count)
// of the largest slot fit in `bits`.
static int sort_passes(const emb_table* t) {
  const int bits = bits_for((unsigned)t->st.max_slot_keys);
  return std::max(1, (bits + kRadixBits - 1) / kRadixBits);
}

// Slot-major placement of the pairs: dest (three scan launches over the bag
// lengths) and the workspace header + sort regions (one launch).
static emb_status launch_placement(const emb_table* t, const int64_t* offsets_d, long long n_bags, long long nnz,
                                   char* ws, const WsLayout& L, cudaStream_t st) {
  WsHeader* hdr = (WsHeader*)(ws + L.hdr);
  unsigned* dest = (unsigned*)(ws + L.dest);
  unsigned* partials = (unsigned*)(ws + L.partials);
  SortSeg* sg = (SortSeg*)(ws + L.sseg);
  const unsigned S = (unsigned)t->st.n_slots;
  const unsigned long long B = (unsigned long long)n_bags / S;
  EMB_CUDA(cudaMemsetAsync(&hdr->total, 0, sizeof(unsigned long long), st));
  if (n_bags > 0) {
    const dim3 grid((unsigned)((B + 31) / 32), (S + 31) / 32);
    len_transpose_kernel<<<grid, 256, 0, st>>>((const long long*)offsets_d, B, S, nnz, dest, hdr);
    EMB_CUDA(launch_scan(dest, dest, (size_t)n_bags, partials, st));
  }
  seg_setup_kernel<<<1, 1024, 0, st>>>(t->view(), hdr, (unsigned)nnz, (unsigned long long)n_bags,
                                       (unsigned)(sort_passes(t) & 1), dest, sg);
  tile_map_kernel<<<(L.n_tiles_sort + 255) / 256, 256, 0, st>>>(sg, L.n_regions, L.n_tiles_sort,
                                                               (unsigned*)(ws + L.treg));
  EMB_CUDA(cudaGetLastError());
  return EMB_OK;
}

// The stable sort of the placed (row, bag) pairs by row, region by region.
// Returns the buffers holding the sorted pairs (A or B by the pass count).
static emb_status sort_placed_pairs(const emb_table* table, int64_t n_bags, unsigned n, char* ws, const WsLayout& L,
                                    cudaStream_t st, unsigned** k_sorted, unsigned** v_sorted) {
  const int passes = sort_passes(table);
  unsigned* counts = (unsigned*)(ws + L.counts);
  unsigned* partials = (unsigned*)(ws + L.partials);
  const size_t smem = scatter_smem();
  EMB_CUDA(cudaFuncSetAttribute(radix_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  unsigned *ki = (unsigned*)(ws + L.kA), *vi = (unsigned*)(ws + L.vA);
  unsigned *ko = (unsigned*)(ws + L.kB), *vo = (unsigned*)(ws + L.vB);
  const SortSeg* sg = (const SortSeg*)(ws + L.sseg);
  const unsigned* treg = (const unsigned*)(ws + L.treg);
  for (int p = 0; p < passes; ++p) {
    const int shift = p * kRadixBits;
    radix_count_kernel<<<L.n_tiles_sort, kSortThreads, 0, st>>>(ki, sg, L.n_regions, shift, counts, treg);
    EMB_CUDA(launch_scan(counts, counts, (size_t)kDigits * L.n_tiles_sort, partials, st));
    radix_scatter_kernel<<<L.n_tiles_sort, kSortThreads, smem, st>>>(ki, vi, ko, vo, shift, counts, sg, L.n_regions,
                                                                     (unsigned)table->st.n_keys, (unsigned)n_bags, treg);
    EMB_CUDA(cudaGetLastError());
    std::swap(ki, ko);
    std::swap(vi, vo);
  }
  *k_sorted = ki;
  *v_sorted = vi;
  return EMB_OK;
}

// The optimizer of one backward call.  The Adagrad entry points serve both
// Adagrad tables (one accumulator per element) and row-wise Adagrad tables
// (one per row); the table's optimizer picks the update.
struct BwdOpt {
  bool ftrl;
  AdagradStep ada;
  FtrlStep fp;
};

static bool opt_fits_table(const emb_table* t, const BwdOpt& o) {
  return o.ftrl ? t->optimizer == EMB_OPT_FTRL
                : (t->optimizer == EMB_OPT_ADAGRAD || t->optimizer == EMB_OPT_ROWWISE_ADAGRAD);
}

// The backward.  With `recorded`, the (row, bag) pairs, 1/L and the header were
// written by emb_lookup_fwd_record (or emb_lookup_fwd_dedup, which also sorted
// them: `presorted`) and those phases are skipped.
static emb_status run_bwd(emb_table* table, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                          int64_t nnz, emb_pool pool, const float* grad_out_d, const BwdOpt& opt, char* ws,
                          const WsLayout& L, cudaStream_t st, bool recorded = false, bool presorted = false) {
  const unsigned n = (unsigned)nnz;
  // grad_out rows are addressed as 32-bit float4 indices
  if ((unsigned long long)(n_bags / table->st.n_slots) * (unsigned long long)table->st.sum_dims >= (1ULL << 34))
    return fail(EMB_ERR_UNSUPPORTED, "grad_out larger than 2^34 elements");
  const int passes = sort_passes(table);
  TableView v = table->view();
  unsigned* kA = (unsigned*)(ws + L.kA);
  unsigned* kB = (unsigned*)(ws + L.kB);
  unsigned* vA = (unsigned*)(ws + L.vA);
  unsigned* vB = (unsigned*)(ws + L.vB);
  float* scale = (float*)(ws + L.scale);
  const int mean = pool == EMB_POOL_MEAN;

  // Every later kernel treats rows >= n_rows and bags >= n_bags as absent
  // (misses, and with malformed offsets every position: see seg_setup_kernel).
  if (!recorded) {
    emb_status rc = launch_placement(table, offsets_d, n_bags, nnz, ws, L, st);
    if (rc != EMB_OK) return rc;
    long long blocks = std::min<long long>((n_bags * 32 + 255) / 256, resident_blocks(256));
    expand_kernel<<<(int)std::max(1LL, blocks), 256, 0, st>>>(v, (const long long*)offsets_d, n_bags,
                                                              (const long long*)keys_d, nnz, mean,
                                                              (const unsigned*)(ws + L.dest), kA, vA, scale);
    EMB_CUDA(cudaGetLastError());
  }
  mark_phase(table, 0, st);
  if (nnz == 0) {
    for (int ph = 1; ph < EMB_BWD_PHASES; ++ph) mark_phase(table, ph, st);
    return EMB_OK;
  }

  unsigned *ki = kA, *vi = vA;
  if (presorted) {
    if (passes & 1) {
      ki = kB;
      vi = vB;
    }
  } else {
    emb_status rc = sort_placed_pairs(table, n_bags, n, ws, L, st, &ki, &vi);
    if (rc != EMB_OK) return rc;
  }
  mark_phase(table, 1, st);
  // ki/vi hold the sorted pairs
  const bool half = table->st.wdtype == EMB_F16;
  const unsigned nb = (unsigned)n_bags;
  cudaError_t e;
  if (opt.ftrl) {
    e = half ? dispatch_reduce<__half>(table, ki, vi, scale, mean, grad_out_d, n, nb, L, ws, opt.fp, st)
             : dispatch_reduce<float>(table, ki, vi, scale, mean, grad_out_d, n, nb, L, ws, opt.fp, st);
  } else if (table->optimizer == EMB_OPT_ROWWISE_ADAGRAD) {
    const RowAdagradStep ro{opt.ada.lr, opt.ada.eps};
    e = half ? dispatch_reduce<__half>(table, ki, vi, scale, mean, grad_out_d, n, nb, L, ws, ro, st)
             : dispatch_reduce<float>(table, ki, vi, scale, mean, grad_out_d, n, nb, L, ws, ro, st);
  } else {
    e = half ? dispatch_reduce<__half>(table, ki, vi, scale, mean, grad_out_d, n, nb, L, ws, opt.ada, st)
             : dispatch_reduce<float>(table, ki, vi, scale, mean, grad_out_d, n, nb, L, ws, opt.ada, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "segmented reduce launch");
  return EMB_OK;
}

// ------------------------------------------------------------------ forward with a within-batch dedupe
//
// The Tencent PCG talk ("各阶段优化详细介绍") deduplicates the keys of a group
// before their rows are moved.  Here the dedupe is the backward's own work
// done first: every occurrence resolved and placed, the pairs sorted by row;
// then each unique row is read from the table once, into registers, and added
// into every bag that holds it.  The sorted pairs stay in the workspace, so
// the recorded backward that follows skips its sort.  A pooled row receives
// adds from many warps, so they are float32 atomics: the output agrees with
// emb_lookup_fwd within rounding but is not bitwise reproducible.
constexpr int kDedupChunk = 64;  // sorted positions per lane group

template <typename TW, int NCB>
__global__ void __launch_bounds__(256) dedup_pool_kernel(TableView t, const unsigned* __restrict__ K,
                                                         const unsigned* __restrict__ V,
                                                         const float* __restrict__ scale, int mean, unsigned n,
                                                         unsigned n_bags, float* __restrict__ out, int G) {
  const int lane = threadIdx.x & 31;
  const int P = 32 / G;
  const int sub = lane / G, li = lane % G;
  const unsigned gid = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * P + sub;
  const unsigned ngroups = ((gridDim.x * blockDim.x) >> 5) * P;
  const unsigned S = (unsigned)t.n_slots, miss = t.n_rows;
  const TW* W = static_cast<const TW*>(t.W);
  for (unsigned long long c0 = (unsigned long long)gid * kDedupChunk; c0 < n;
       c0 += (unsigned long long)ngroups * kDedupChunk) {
    const unsigned c1 = (unsigned)min(c0 + kDedupChunk, (unsigned long long)n);
    unsigned cur = kNoRow;
    RowGeo g{0, 0, 0, false};
    float w[NCB][4];
    for (unsigned i = (unsigned)c0; i < c1; ++i) {
      const unsigned row = K[i], bag = V[i];
      if (row >= miss || bag >= n_bags) continue;
      if (row != cur) {  // a new run: its row is read from the table once
        cur = row;
        g = geo_from_slot(t, row, (int)(bag % S));
#pragma unroll
        for (int cc = 0; cc < NCB; ++cc) {
          const int ce = (cc * G + li) * 4;
          if (g.ok && ce < g.D) {
            ldw4(W + g.e0 + ce, w[cc]);
          } else {
            w[cc][0] = w[cc][1] = w[cc][2] = w[cc][3] = 0.f;
          }
        }
      }
      if (!g.ok) continue;
      const float sc = mean ? scale[bag] : 1.f;
      float* o = out + (size_t)(bag / S) * (unsigned)t.sum_dims + (unsigned)g.col;
#pragma unroll
      for (int cc = 0; cc < NCB; ++cc) {
        const int ce = (cc * G + li) * 4;
        if (ce < g.D)
          atomicAdd(reinterpret_cast<float4*>(o + ce),
                    make_float4(w[cc][0] * sc, w[cc][1] * sc, w[cc][2] * sc, w[cc][3] * sc));
      }
    }
  }
}

template <typename TW>
static cudaError_t launch_dedup_pool(const emb_table* t, const unsigned* K, const unsigned* V, const float* scale,
                                     int mean, unsigned n, unsigned n_bags, float* out, cudaStream_t st) {
  const int vecs = (t->st.max_dim + 3) / 4;  // 4-float column vectors of the widest row
  int G = 1;
  while (G < vecs && G < 32) G <<= 1;
  const int ncb = (vecs + G - 1) / G;
  const unsigned groups = (n + kDedupChunk - 1) / kDedupChunk;
  const long long blocks =
      std::max(1LL, std::min<long long>(((long long)groups * G + 255) / 256, (long long)sm_count() * 8));
  TableView v = t->fwd_view();  // master-copy tables: the f16 copy, as the forward reads
  if (ncb <= 1)
    dedup_pool_kernel<TW, 1><<<(int)blocks, 256, 0, st>>>(v, K, V, scale, mean, n, n_bags, out, G);
  else if (ncb <= 2)
    dedup_pool_kernel<TW, 2><<<(int)blocks, 256, 0, st>>>(v, K, V, scale, mean, n, n_bags, out, G);
  else
    dedup_pool_kernel<TW, 4><<<(int)blocks, 256, 0, st>>>(v, K, V, scale, mean, n, n_bags, out, G);
  return cudaGetLastError();
}

// Scratch for emb_bwd_adagrad_noalloc, for callers that cannot allocate
// device memory.  The loader reserves it on every GPU that loads this library;
// host code must not pass the symbol itself to a kernel (on the host it only
// names a stand-in), so its device address is looked up with
// cudaGetSymbolAddress, once per CUDA context: a context that is destroyed
// (cudaDeviceReset) and created again reloads the module, and the array may
// then sit at another address, so the cache is keyed by the context's
// unique id, not by the device index.
static __device__ __align__(256) unsigned char g_noalloc_scratch[EMB_NOALLOC_SCRATCH_BYTES];

typedef int (*CtxGetCurrentFn)(void** ctx);
typedef int (*CtxGetIdFn)(void* ctx, unsigned long long* id);

static std::mutex g_noalloc_mu;
static std::vector<std::pair<unsigned long long, void*>> g_noalloc_ptr;  // (context id, scratch address)

// Unique id of the calling thread's current context (0 if none is current),
// through the driver entry points the runtime hands out (the library links
// no driver library directly).
static emb_status current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", (void**)&get_cur, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      get_cur = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", (void**)&get_id, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      get_id = nullptr;
    cudaGetLastError();
  });
  if (!get_cur || !get_id) return fail(EMB_ERR_CUDA, "driver entry points cuCtxGetCurrent/cuCtxGetId unavailable");
  void* ctx = nullptr;
  if (get_cur(&ctx) != 0) return fail(EMB_ERR_CUDA, "cuCtxGetCurrent failed");
  *id = 0;
  if (ctx && get_id(ctx, id) != 0) return fail(EMB_ERR_CUDA, "cuCtxGetId failed");
  return EMB_OK;
}

static emb_status noalloc_scratch(void** out) {
  unsigned long long id = 0;
  emb_status rc = current_context_id(&id);
  if (rc != EMB_OK) return rc;
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  if (id != 0)
    for (const auto& e : g_noalloc_ptr)
      if (e.first == id) {
        *out = e.second;
        return EMB_OK;
      }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // also makes the device's context current
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
  if (id == 0 && (rc = current_context_id(&id)) != EMB_OK) return rc;
  if (id != 0) g_noalloc_ptr.emplace_back(id, p);
  *out = p;
  return EMB_OK;
}

}  // namespace emb

using namespace emb;

extern "C" {

emb_status emb_bwd_adagrad_noalloc(emb_table* table, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                                   int64_t nnz, emb_pool pool, const float* grad_out_d, float lr, float eps,
                                   void* stream) {
  emb_status rc = check_batch(table, offsets_d, n_bags, keys_d, nnz, pool);
  if (rc != EMB_OK) return rc;
  if (!opt_fits_table(table, BwdOpt{false, {lr, eps}, {}}))
    return fail(EMB_ERR_INVALID_ARG, "the table's optimizer is not Adagrad");
  if (n_bags > 0 && !grad_out_d) return fail(EMB_ERR_INVALID_ARG, "grad_out is NULL");
  if (((uintptr_t)grad_out_d & 15) != 0) return fail(EMB_ERR_INVALID_ARG, "grad_out must be 16-byte aligned");
  const WsLayout L = ws_layout(table, n_bags, nnz);
  if (L.total > (size_t)EMB_NOALLOC_SCRATCH_BYTES) {
    char buf[192];
    std::snprintf(buf, sizeof buf,
                  "batch needs %zu bytes of scratch; emb_bwd_adagrad_noalloc holds %u (use emb_bwd_adagrad "
                  "with a workspace)", L.total, (unsigned)EMB_NOALLOC_SCRATCH_BYTES);
    return fail(EMB_ERR_UNSUPPORTED, buf);
  }
  void* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch)) != EMB_OK) return rc;
  return run_bwd(table, offsets_d, n_bags, keys_d, nnz, pool, grad_out_d, BwdOpt{false, {lr, eps}, {}},
                 (char*)scratch, L, (cudaStream_t)stream);
}

emb_status emb_lookup_fwd_record(emb_table* table, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                                 int64_t nnz, emb_pool pool, float* out_d, void* workspace_d, size_t ws_bytes,
                                 void* stream) {
  emb_status rc = check_batch(table, offsets_d, n_bags, keys_d, nnz, pool);
  if (rc != EMB_OK) return rc;
  if (n_bags > 0 && !out_d) return fail(EMB_ERR_INVALID_ARG, "out is NULL");
  if (((uintptr_t)out_d & 15) != 0) return fail(EMB_ERR_INVALID_ARG, "out must be 16-byte aligned");
  const WsLayout L = ws_layout(table, n_bags, nnz);
  if (!workspace_d || ws_bytes < L.total) return fail(EMB_ERR_WORKSPACE, "workspace missing or too small");
  if (((uintptr_t)workspace_d & 255) != 0) return fail(EMB_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  char* ws = (char*)workspace_d;
  if ((rc = launch_placement(table, offsets_d, n_bags, nnz, ws, L, st)) != EMB_OK) return rc;
  if (n_bags > 0) {
    // bags are handed out in order from a counter (measured 17.7 -> 15.1 ms at
    // 100M keys x dim 128 against a static order; Zipf bag lengths unbalance it)
    unsigned long long* fwork = (unsigned long long*)(ws + L.fwork);
    EMB_CUDA(cudaMemsetAsync(fwork, 0, sizeof(unsigned long long), st));
    cudaError_t e = launch_forward(table, (const long long*)offsets_d, n_bags, (const long long*)keys_d, nnz,
                                   pool == EMB_POOL_MEAN, out_d, (unsigned*)(ws + L.kA), (unsigned*)(ws + L.vA),
                                   (float*)(ws + L.scale), (const unsigned*)(ws + L.dest),
                                   &((const WsHeader*)(ws + L.hdr))->placed, fwork, st);
    if (e != cudaSuccess) return cuda_fail(e, "fwd_pool_kernel launch");
  }
  EMB_CUDA(cudaGetLastError());
  table->rec_ws = workspace_d;
  table->rec_nnz = nnz;
  table->rec_bags = n_bags;
  table->rec_pool = (int)pool;
  table->rec_sorted = false;
  return EMB_OK;
}

// The recorded backward with either optimizer.
static emb_status bwd_recorded(emb_table* table, int64_t n_bags, int64_t nnz, emb_pool pool, const float* grad_out_d,
                               const BwdOpt& opt, void* workspace_d, size_t ws_bytes, void* stream) {
  if (!table) return fail(EMB_ERR_INVALID_ARG, "table is NULL");
  if (!opt_fits_table(table, opt))
    return fail(EMB_ERR_INVALID_ARG, "the table was created for another optimizer");
  if (!workspace_d || workspace_d != table->rec_ws || nnz != table->rec_nnz || n_bags != table->rec_bags ||
      (int)pool != table->rec_pool)
    return fail(EMB_ERR_INVALID_ARG, "no emb_lookup_fwd_record of this batch shape in this workspace");
  if (n_bags > 0 && !grad_out_d) return fail(EMB_ERR_INVALID_ARG, "grad_out is NULL");
  if (((uintptr_t)grad_out_d & 15) != 0) return fail(EMB_ERR_INVALID_ARG, "grad_out must be 16-byte aligned");
  const WsLayout L = ws_layout(table, n_bags, nnz);
  if (ws_bytes < L.total) return fail(EMB_ERR_WORKSPACE, "workspace missing or too small");
  return run_bwd(table, nullptr, n_bags, nullptr, nnz, pool, grad_out_d, opt, (char*)workspace_d, L,
                 (cudaStream_t)stream, true, table->rec_sorted);
}

// The backward with a caller workspace and either optimizer.
static emb_status bwd_workspace(emb_table* table, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                                int64_t nnz, emb_pool pool, const float* grad_out_d, const BwdOpt& opt,
                                void* workspace_d, size_t ws_bytes, void* stream) {
  emb_status rc = check_batch(table, offsets_d, n_bags, keys_d, nnz, pool);
  if (rc != EMB_OK) return rc;
  if (!opt_fits_table(table, opt))
    return fail(EMB_ERR_INVALID_ARG, "the table was created for another optimizer");
  if (n_bags > 0 && !grad_out_d) return fail(EMB_ERR_INVALID_ARG, "grad_out is NULL");
  if (((uintptr_t)grad_out_d & 15) != 0) return fail(EMB_ERR_INVALID_ARG, "grad_out must be 16-byte aligned");
  const WsLayout L = ws_layout(table, n_bags, nnz);
  if (!workspace_d || ws_bytes < L.total) return fail(EMB_ERR_WORKSPACE, "workspace missing or too small");
  if (((uintptr_t)workspace_d & 255) != 0) return fail(EMB_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  return run_bwd(table, offsets_d, n_bags, keys_d, nnz, pool, grad_out_d, opt, (char*)workspace_d, L,
                 (cudaStream_t)stream);
}

static emb_status ftrl_opt(const emb_ftrl_params* p, BwdOpt* o) {
  if (!p) return fail(EMB_ERR_INVALID_ARG, "FTRL parameters are NULL");
  if (!(p->alpha > 0.f) || !(p->beta >= 0.f) || !(p->lambda1 >= 0.f) || !(p->lambda2 >= 0.f))
    return fail(EMB_ERR_INVALID_ARG, "FTRL needs alpha > 0 and beta, lambda1, lambda2 >= 0");
  *o = BwdOpt{true, {}, {p->alpha, p->beta, p->lambda1, p->lambda2}};
  return EMB_OK;
}

emb_status emb_lookup_fwd_dedup(emb_table* table, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                                int64_t nnz, emb_pool pool, float* out_d, void* workspace_d, size_t ws_bytes,
                                void* stream) {
  emb_status rc = check_batch(table, offsets_d, n_bags, keys_d, nnz, pool);
  if (rc != EMB_OK) return rc;
  if (n_bags > 0 && !out_d) return fail(EMB_ERR_INVALID_ARG, "out is NULL");
  if (((uintptr_t)out_d & 15) != 0) return fail(EMB_ERR_INVALID_ARG, "out must be 16-byte aligned");
  const WsLayout L = ws_layout(table, n_bags, nnz);
  if (!workspace_d || ws_bytes < L.total) return fail(EMB_ERR_WORKSPACE, "workspace missing or too small");
  if (((uintptr_t)workspace_d & 255) != 0) return fail(EMB_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  char* ws = (char*)workspace_d;
  const int mean = pool == EMB_POOL_MEAN;
  if ((rc = launch_placement(table, offsets_d, n_bags, nnz, ws, L, st)) != EMB_OK) return rc;
  unsigned* kA = (unsigned*)(ws + L.kA);
  unsigned* vA = (unsigned*)(ws + L.vA);
  float* scale = (float*)(ws + L.scale);
  if (n_bags > 0) {
    const long long blocks = std::min<long long>((n_bags * 32 + 255) / 256, resident_blocks(256));
    expand_kernel<<<(int)std::max(1LL, blocks), 256, 0, st>>>(table->fwd_view(), (const long long*)offsets_d,
                                                              n_bags, (const long long*)keys_d, nnz, mean,
                                                              (const unsigned*)(ws + L.dest), kA, vA, scale);
    EMB_CUDA(cudaGetLastError());
    EMB_CUDA(cudaMemsetAsync(out_d, 0, (size_t)(n_bags / table->st.n_slots) * (size_t)table->st.sum_dims * 4, st));
  }
  if (nnz > 0) {
    unsigned *ki, *vi;
    if ((rc = sort_placed_pairs(table, n_bags, (unsigned)nnz, ws, L, st, &ki, &vi)) != EMB_OK) return rc;
    cudaError_t e = table->fwd_half()
                        ? launch_dedup_pool<__half>(table, ki, vi, scale, mean, (unsigned)nnz, (unsigned)n_bags,
                                                    out_d, st)
                        : launch_dedup_pool<float>(table, ki, vi, scale, mean, (unsigned)nnz, (unsigned)n_bags,
                                                   out_d, st);
    if (e != cudaSuccess) return cuda_fail(e, "dedup_pool_kernel launch");
  }
  table->rec_ws = workspace_d;
  table->rec_nnz = nnz;
  table->rec_bags = n_bags;
  table->rec_pool = (int)pool;
  table->rec_sorted = true;
  return EMB_OK;
}

emb_status emb_bwd_adagrad_recorded(emb_table* table, int64_t n_bags, int64_t nnz, emb_pool pool,
                                    const float* grad_out_d, float lr, float eps, void* workspace_d, size_t ws_bytes,
                                    void* stream) {
  return bwd_recorded(table, n_bags, nnz, pool, grad_out_d, BwdOpt{false, {lr, eps}, {}}, workspace_d, ws_bytes,
                      stream);
}

emb_status emb_bwd_ftrl_recorded(emb_table* table, int64_t n_bags, int64_t nnz, emb_pool pool,
                                 const float* grad_out_d, const emb_ftrl_params* params, void* workspace_d,
                                 size_t ws_bytes, void* stream) {
  BwdOpt o;
  emb_status rc = ftrl_opt(params, &o);
  if (rc != EMB_OK) return rc;
  return bwd_recorded(table, n_bags, nnz, pool, grad_out_d, o, workspace_d, ws_bytes, stream);
}

emb_status emb_bwd_ftrl(emb_table* table, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                        int64_t nnz, emb_pool pool, const float* grad_out_d, const emb_ftrl_params* params,
                        void* workspace_d, size_t ws_bytes, void* stream) {
  BwdOpt o;
  emb_status rc = ftrl_opt(params, &o);
  if (rc != EMB_OK) return rc;
  return bwd_workspace(table, offsets_d, n_bags, keys_d, nnz, pool, grad_out_d, o, workspace_d, ws_bytes, stream);
}

emb_status emb_bwd_phase_events(emb_table* table, void* const* events, int n) {
  if (!table || n < 0 || n > EMB_BWD_PHASES || (n > 0 && !events))
    return fail(EMB_ERR_INVALID_ARG, "bad phase events");
  for (int i = 0; i < EMB_BWD_PHASES; ++i) table->phase_events[i] = i < n ? events[i] : nullptr;
  table->n_phase_events = n;
  return EMB_OK;
}

emb_status emb_bwd_workspace_size(const emb_table* table, int64_t n_bags, int64_t nnz, size_t* bytes) {
  if (!table || !bytes || n_bags < 0 || nnz < 0) return fail(EMB_ERR_INVALID_ARG, "bad workspace query");
  if (n_bags > EMB_MAX_BAGS || nnz > EMB_MAX_NNZ) return fail(EMB_ERR_UNSUPPORTED, "batch exceeds EMB_MAX_* limits");
  *bytes = ws_layout(table, n_bags, nnz).total;
  return EMB_OK;
}

emb_status emb_bwd_adagrad(emb_table* table, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                           int64_t nnz, emb_pool pool, const float* grad_out_d, float lr, float eps,
                           void* workspace_d, size_t ws_bytes, void* stream) {
  return bwd_workspace(table, offsets_d, n_bags, keys_d, nnz, pool, grad_out_d, BwdOpt{false, {lr, eps}, {}},
                       workspace_d, ws_bytes, stream);
}

emb_status emb_bwd_unique_keys(const emb_table* table, const void* workspace_d, size_t ws_bytes, int64_t* keys_out_d,
                               int64_t* n_unique_d, void* stream) {
  if (!table || !workspace_d || !keys_out_d || !n_unique_d) return fail(EMB_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t st = (cudaStream_t)stream;
  WsHeader h;
  EMB_CUDA(cudaStreamSynchronize(st));
  EMB_CUDA(cudaMemcpy(&h, workspace_d, sizeof h, cudaMemcpyDeviceToHost));
  if (h.magic != kMagic) return fail(EMB_ERR_WORKSPACE, "workspace holds no backward result");
  const WsLayout L = ws_layout(table, h.n_bags, h.nnz);
  if (ws_bytes < L.total) return fail(EMB_ERR_WORKSPACE, "workspace smaller than the backward that filled it");
  char* ws = (char*)const_cast<void*>(workspace_d);
  const unsigned* K = (const unsigned*)(ws + (h.sorted_in_b ? L.kB : L.kA));
  unsigned* partials = (unsigned*)(ws + L.partials);
  const size_t n = h.nnz;
  const unsigned np = (unsigned)std::max<size_t>(1, (n + kScanTile - 1) / kScanTile);
  if (n == 0) {
    EMB_CUDA(cudaMemsetAsync(partials, 0, 8, st));
  } else {
    head_count_kernel<<<np, kScanThreads, 0, st>>>(K, n, h.miss_row, partials);
    scan_partials_kernel<<<1, 1024, 0, st>>>(partials, np);
    head_write_kernel<<<np, kScanThreads, 0, st>>>(K, n, h.miss_row, partials, table->row_key_d,
                                                   (long long*)keys_out_d);
  }
  store_count_kernel<<<1, 1, 0, st>>>(partials, n == 0 ? 0 : np, (long long*)n_unique_d, (WsHeader*)ws);
  EMB_CUDA(cudaGetLastError());
  return EMB_OK;
}

}  // extern "C"
