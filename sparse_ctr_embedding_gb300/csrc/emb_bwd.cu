// Backward: duplicate-key gradient reduction + element-wise sparse Adagrad.
//
// Tencent PCG DataFun talk, "计算优化": one backward kernel updates every
// feature of the unified table.  JD ads article, 3.2.1: Adagrad keeps a
// per-parameter sum of squared gradients, updates element-wise, and leaves
// features that are absent from the batch untouched.
//
// Pipeline (all on the caller's stream, no host synchronisation):
//  1. expand    one warp per bag: probe each key; emit the pair
//               (internal row, bag) per occurrence (row = n_rows for a miss,
//               which sorts last) and, for mean, 1/L per bag.
//  2. sort      stable LSD radix sort of the pairs by row (hand-written:
//               per-tile digit counts, a device-wide scan, then a stable
//               scatter ranked with warp match/ballot and staged in shared
//               memory so every digit run is written contiguously).
//               Rows are numbered slot-major, so the sorted order walks one
//               feature slot (one column block of grad_out) at a time.
//  3. reduce    the sorted positions are cut into chunks of kChunk; one warp
//               per chunk.  Every run of equal rows inside a chunk ("piece")
//               is summed in float32, in sorted order (so in occurrence
//               order: the sort is stable), by a group of G lanes.  A piece
//               that is a whole segment (all occurrences of its row) applies
//               Adagrad to the row directly.  A piece cut by a chunk edge
//               leaves a partial sum: the head piece of a segment in slot A
//               of its chunk, later pieces in slot B of theirs.
//  4. fixup     one warp per segment that spans chunks: A + B + B ... in
//               chunk order (a fixed tree across the warp's lane groups),
//               then Adagrad.
// No float atomics: every sum has a fixed order, so the step is bitwise
// reproducible.  The Adagrad arithmetic per element, in float32:
//   g = G;  acc += g * g;  w -= lr * g / (sqrt(acc) + eps)
// with IEEE sqrt and division (no fast-math), half weights rounded to
// nearest-even on store.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "emb_internal.cuh"

namespace emb {

emb_status check_batch(const emb_table* t, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                       int64_t nnz, int pool);

constexpr int kChunk = 256;                      // sorted positions per reduce chunk
constexpr int kSortWarps = 8;
constexpr int kSortThreads = kSortWarps * 32;
constexpr int kSortItems = 16;                   // keys per lane per tile
constexpr int kSortTile = kSortThreads * kSortItems;
constexpr int kRadixBits = 8;
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
  unsigned sorted_in_b;  // 1: sorted pairs are in buffer B
  unsigned miss_row;     // sentinel row of a miss (= n_rows)
  unsigned n_unique;     // filled by emb_bwd_unique_keys
};

static size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
  size_t hdr, kA, kB, vA, vB, scale, counts, partials, partA, partB, arow, uniq, total;
  unsigned n_tiles_sort, n_chunks, n_scan_partials;
  int max_dim;
};

static WsLayout ws_layout(const emb_table* t, long long n_bags, long long nnz) {
  WsLayout L{};
  const size_t n = (size_t)std::max<long long>(nnz, 1);
  L.max_dim = t->st.max_dim;
  L.n_tiles_sort = (unsigned)((n + kSortTile - 1) / kSortTile);
  L.n_chunks = (unsigned)((n + kChunk - 1) / kChunk);
  const size_t n_counts = (size_t)kDigits * L.n_tiles_sort;
  const size_t scan_n = std::max(n_counts, n);
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
  L.scale = take((size_t)std::max<long long>(n_bags, 1) * 4);
  L.counts = take(n_counts * 4);
  L.partials = take((size_t)(L.n_scan_partials + 1) * 4);
  L.partA = take((size_t)L.n_chunks * L.max_dim * 4);
  L.partB = take((size_t)L.n_chunks * L.max_dim * 4);
  L.arow = take((size_t)L.n_chunks * 4);
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

__global__ void __launch_bounds__(256) expand_kernel(TableView t, const long long* __restrict__ offsets,
                                                     long long n_bags, const long long* __restrict__ keys,
                                                     long long nnz, int mean, unsigned* __restrict__ K,
                                                     unsigned* __restrict__ V, float* __restrict__ scale,
                                                     WsHeader* hdr, unsigned sorted_in_b) {
  const int lane = threadIdx.x & 31;
  const long long gw = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  if (gw == 0 && lane == 0) {
    hdr->magic = kMagic;
    hdr->nnz = (unsigned)nnz;
    hdr->n_bags = (unsigned)n_bags;
    hdr->sorted_in_b = sorted_in_b;
    hdr->miss_row = t.n_rows;
    hdr->n_unique = 0;
  }
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const unsigned S = (unsigned)t.n_slots;
  for (long long bag = gw; bag < n_bags; bag += nwarps) {
    const int s = (int)((unsigned)bag % S);
    long long start = offsets[bag], end = offsets[bag + 1];
    if (start < 0 || end > nnz || end < start || (bag == 0 && start != 0) || (bag == n_bags - 1 && end != nnz)) {
      if (lane == 0) atomicOr(t.flags, EMB_FLAG_BAD_OFFSETS);
      start = min(max(start, 0LL), nnz);
      end = min(max(end, start), nnz);
    }
    if (mean && lane == 0) scale[bag] = end > start ? 1.0f / (float)(end - start) : 0.f;
    for (long long i = start + lane; i < end; i += 32) {
      const long long k = keys[i];
      unsigned row = t.n_rows, ext;
      unsigned long long h;
      if (key_slot(k) != s) {
        atomicOr(t.flags, EMB_FLAG_SLOT_MISMATCH);
      } else if (!probe(t, k, &row, &ext, &h)) {
        row = t.n_rows;
      }
      K[i] = row;
      V[i] = (unsigned)bag;
    }
  }
}

// ------------------------------------------------------------------ 2. radix sort

// Per-warp digit counting over one tile: each warp walks its 32*kSortItems
// consecutive keys in order, 32 at a time; lanes holding the same digit are
// grouped with __match_any_sync and the group leader bumps the warp's counter.
// Returns, per item, its rank among equal digits of this warp (stable).
__device__ __forceinline__ void warp_rank(unsigned (&d)[kSortItems], unsigned (&rank)[kSortItems], bool (&valid)[kSortItems],
                                          unsigned* cnt /* this warp's kDigits counters */) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < kSortItems; ++r) {
    const unsigned key = valid[r] ? d[r] : 0xFFFFFFFFu;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int leader = __ffs(peers) - 1;
    unsigned base = 0;
    if (valid[r] && lane == leader) {
      base = cnt[d[r]];
      cnt[d[r]] = base + __popc(peers);
    }
    base = __shfl_sync(0xffffffffu, base, leader);
    rank[r] = base + __popc(peers & lanemask_lt());
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kSortThreads) radix_count_kernel(const unsigned* __restrict__ keys, unsigned n,
                                                                   int shift, unsigned* __restrict__ counts,
                                                                   unsigned n_tiles) {
  __shared__ unsigned cnt[kSortWarps][kDigits];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kSortWarps * kDigits; i += kSortThreads) (&cnt[0][0])[i] = 0;
  __syncthreads();
  const unsigned tile = blockIdx.x;
  const unsigned base = tile * kSortTile + w * 32 * kSortItems;
  unsigned d[kSortItems], rank[kSortItems];
  bool valid[kSortItems];
#pragma unroll
  for (int r = 0; r < kSortItems; ++r) {
    const unsigned i = base + r * 32 + lane;
    valid[r] = i < n;
    d[r] = valid[r] ? (keys[i] >> shift) & (kDigits - 1) : 0;
  }
  warp_rank(d, rank, valid, cnt[w]);
  __syncthreads();
  for (int dg = threadIdx.x; dg < kDigits; dg += kSortThreads) {
    unsigned tot = 0;
#pragma unroll
    for (int ww = 0; ww < kSortWarps; ++ww) tot += cnt[ww][dg];
    counts[(size_t)dg * n_tiles + tile] = tot;
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

__global__ void __launch_bounds__(kSortThreads) radix_scatter_kernel(
    const unsigned* __restrict__ kin, const unsigned* __restrict__ vin, unsigned* __restrict__ kout,
    unsigned* __restrict__ vout, unsigned n, int shift, const unsigned* __restrict__ counts, unsigned n_tiles) {
  extern __shared__ unsigned smem[];
  unsigned(*cnt)[kDigits] = reinterpret_cast<unsigned(*)[kDigits]>(smem);  // [kSortWarps][kDigits]
  unsigned* gbase = smem + kSortWarps * kDigits;                             // [kDigits]
  unsigned* bstart = gbase + kDigits;                                         // [kDigits]
  unsigned* wtot = bstart + kDigits;                                          // [33]
  unsigned* tk = wtot + 33;                                                   // [kSortTile]
  unsigned* tv = tk + kSortTile;                                              // [kSortTile]
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned tile = blockIdx.x;
  for (int i = threadIdx.x; i < kSortWarps * kDigits; i += kSortThreads) smem[i] = 0;
  for (int dg = threadIdx.x; dg < kDigits; dg += kSortThreads) gbase[dg] = counts[(size_t)dg * n_tiles + tile];
  __syncthreads();
  const unsigned base = tile * kSortTile + w * 32 * kSortItems;
  unsigned k[kSortItems], v[kSortItems], d[kSortItems], rank[kSortItems];
  bool valid[kSortItems];
#pragma unroll
  for (int r = 0; r < kSortItems; ++r) {
    const unsigned i = base + r * 32 + lane;
    valid[r] = i < n;
    k[r] = valid[r] ? kin[i] : 0;
    v[r] = valid[r] ? vin[i] : 0;
    d[r] = (k[r] >> shift) & (kDigits - 1);
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
      bstart[dg] = excl;
#pragma unroll
      for (int ww = 0; ww < kSortWarps; ++ww) cnt[ww][dg] += excl;
      excl += run[j];
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kSortItems; ++r) {
    if (valid[r]) {
      const unsigned pos = cnt[w][d[r]] + rank[r];
      tk[pos] = k[r];
      tv[pos] = v[r];
    }
  }
  __syncthreads();
  const unsigned tile_n = min((unsigned)kSortTile, n - tile * kSortTile);
  for (unsigned j = threadIdx.x; j < tile_n; j += kSortThreads) {
    const unsigned kk = tk[j];
    const unsigned dg = (kk >> shift) & (kDigits - 1);
    const unsigned gp = gbase[dg] + (j - bstart[dg]);
    kout[gp] = kk;
    vout[gp] = tv[j];
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
  unsigned v[kScanItems];
  unsigned s = 0;
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    v[j] = base + j < n ? in[base + j] : 0;
    s += v[j];
  }
  unsigned excl = block_excl_scan(s, wt) + partials[blockIdx.x];
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    if (base + j < n) out[base + j] = excl;
    excl += v[j];
  }
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
__device__ __forceinline__ void stw4(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void stw4(__half* p, const float (&v)[4]) {
  const __half2 a = __floats2half2_rn(v[0], v[1]);  // round-to-nearest-even
  const __half2 b = __floats2half2_rn(v[2], v[3]);
  uint2 x;
  x.x = *reinterpret_cast<const unsigned*>(&a);
  x.y = *reinterpret_cast<const unsigned*>(&b);
  *reinterpret_cast<uint2*>(p) = x;
}

// Element-wise Adagrad on one lane's columns of one row.
template <typename TW, int NCB>
__device__ __forceinline__ void adagrad_row(const TableView& t, long long e0, int D, int G, int li,
                                            const float (&g)[NCB][4], float lr, float eps) {
  TW* W = static_cast<TW*>(t.W);
#pragma unroll
  for (int c = 0; c < NCB; ++c) {
    const int ce = (c * G + li) * 4;
    if (ce < D) {
      const float4 a = *reinterpret_cast<const float4*>(t.ACC + e0 + ce);
      float av[4] = {a.x, a.y, a.z, a.w};
      float wv[4];
      ldw4(W + e0 + ce, wv);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float gj = g[c][j];
        av[j] = av[j] + gj * gj;
        wv[j] = wv[j] - (lr * gj) / (sqrtf(av[j]) + eps);
      }
      *reinterpret_cast<float4*>(t.ACC + e0 + ce) = make_float4(av[0], av[1], av[2], av[3]);
      stw4(W + e0 + ce, wv);
    }
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

template <typename TW, int G, int NCB, int U>
__global__ void __launch_bounds__(256) segreduce_adagrad_kernel(
    TableView t, const unsigned* __restrict__ K, const unsigned* __restrict__ V, const float* __restrict__ scale,
    int mean, const float* __restrict__ grad, unsigned n, unsigned n_bags, unsigned n_chunks, float* __restrict__ partA,
    float* __restrict__ partB, unsigned* __restrict__ arow, float lr, float eps) {
  constexpr int P = 32 / G;
  __shared__ unsigned piece_start[8][kChunk + 1];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / G, li = lane % G;
  const unsigned miss = t.n_rows;
  const unsigned S = (unsigned)t.n_slots;
  const int maxd = t.max_dim;
  unsigned* ps = piece_start[w];
  const unsigned nwarps = (gridDim.x * blockDim.x) >> 5;
  for (unsigned c = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; c < n_chunks; c += nwarps) {
    const unsigned cs = c * kChunk;
    const unsigned ce = min(cs + kChunk, n);
    // piece starts: cs and every position where the row changes
    unsigned np = 0;
    unsigned prev = cs > 0 ? K[cs - 1] : kNoRow;
    for (unsigned j0 = cs; j0 < ce; j0 += 32) {
      const unsigned i = j0 + lane;
      const unsigned k = i < ce ? K[i] : kNoRow;
      unsigned kp = __shfl_up_sync(0xffffffffu, k, 1);
      if (lane == 0) kp = prev;
      prev = __shfl_sync(0xffffffffu, k, 31);
      const bool st = i < ce && (i == cs || k != kp);
      const unsigned m = __ballot_sync(0xffffffffu, st);
      if (st) ps[np + __popc(m & lanemask_lt())] = i;
      np += __popc(m);
    }
    if (lane == 0) ps[np] = ce;
    if (lane == 0) arow[c] = kNoRow;
    __syncwarp();
    const bool first_starts = cs == 0 || K[cs - 1] != K[cs];
    const bool last_ends = ce >= n || K[ce] != K[ce - 1];
    for (unsigned p = sub; p < np; p += P) {
      const unsigned a = ps[p], b = ps[p + 1];
      const unsigned row = K[a];
      if (row >= miss) continue;  // misses (and anything past the table) sort last
      int D, col;
      long long e0;
      row_geom(t, row, D, col, e0);
      float acc[NCB][4];
#pragma unroll
      for (int cc = 0; cc < NCB; ++cc)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[cc][j] = 0.f;
      for (unsigned i0 = a; i0 < b; i0 += U) {
        float4 gv[U][NCB];
        float sc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const unsigned i = i0 + u;
          unsigned bag = i < b ? V[i] : 0;
          const bool ok = i < b && bag < n_bags;
          bag = ok ? bag : 0;
          sc[u] = ok ? (mean ? scale[bag] : 1.f) : 0.f;
          const float* gp = grad + (size_t)(bag / S) * t.sum_dims + col;
#pragma unroll
          for (int cc = 0; cc < NCB; ++cc) {
            const int cidx = (cc * G + li) * 4;
            gv[u][cc] = (ok && cidx < D) ? __ldg(reinterpret_cast<const float4*>(gp + cidx))
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (i0 + u < b) {
#pragma unroll
            for (int cc = 0; cc < NCB; ++cc) {
              acc[cc][0] += sc[u] * gv[u][cc].x;
              acc[cc][1] += sc[u] * gv[u][cc].y;
              acc[cc][2] += sc[u] * gv[u][cc].z;
              acc[cc][3] += sc[u] * gv[u][cc].w;
            }
          }
        }
      }
      const bool starts = p > 0 || first_starts;
      const bool ends = p + 1 < np || last_ends;
      if (starts && ends) {
        adagrad_row<TW, NCB>(t, e0, D, G, li, acc, lr, eps);
      } else {
        float* dst = (starts ? partA : partB) + (size_t)c * maxd;
        if (starts && li == 0) arow[c] = row;
#pragma unroll
        for (int cc = 0; cc < NCB; ++cc) {
          const int cidx = (cc * G + li) * 4;
          if (cidx < D)
            *reinterpret_cast<float4*>(dst + cidx) = make_float4(acc[cc][0], acc[cc][1], acc[cc][2], acc[cc][3]);
        }
      }
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ 4. fixup of spanning segments

template <typename TW, int G, int NCB>
__global__ void __launch_bounds__(256) fixup_kernel(TableView t, const unsigned* __restrict__ K, unsigned n,
                                                    unsigned n_chunks, const float* __restrict__ partA,
                                                    const float* __restrict__ partB,
                                                    const unsigned* __restrict__ arow, float lr, float eps) {
  constexpr int P = 32 / G;
  const int lane = threadIdx.x & 31;
  const int sub = lane / G, li = lane % G;
  const int maxd = t.max_dim;
  const unsigned nwarps = (gridDim.x * blockDim.x) >> 5;
  for (unsigned c = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; c < n_chunks; c += nwarps) {
    const unsigned row = arow[c];
    if (row >= t.n_rows || c + 1 >= n_chunks) continue;
    // last chunk whose first position still holds this row (K is sorted)
    unsigned lo = c + 1, hi = n_chunks - 1;
    while (lo < hi) {
      const unsigned mid = lo + (hi - lo + 1) / 2;
      if (K[(size_t)mid * kChunk] == row) lo = mid; else hi = mid - 1;
    }
    const unsigned c1 = lo;  // partials: A[c], B[c+1..c1]
    int D, col;
    long long e0;
    row_geom(t, row, D, col, e0);
    const unsigned m = c1 - c + 1;
    const unsigned per = (m + P - 1) / P;
    const unsigned j0 = sub * per, j1 = min(m, j0 + per);
    float acc[NCB][4];
#pragma unroll
    for (int cc = 0; cc < NCB; ++cc)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[cc][j] = 0.f;
    for (unsigned j = j0; j < j1; ++j) {
      const float* src = (j == 0 ? partA + (size_t)c * maxd : partB + (size_t)(c + j) * maxd);
#pragma unroll
      for (int cc = 0; cc < NCB; ++cc) {
        const int cidx = (cc * G + li) * 4;
        if (cidx < D) {
          const float4 x = *reinterpret_cast<const float4*>(src + cidx);
          acc[cc][0] += x.x;
          acc[cc][1] += x.y;
          acc[cc][2] += x.z;
          acc[cc][3] += x.w;
        }
      }
    }
    // groups hold consecutive ranges: combine with a fixed xor tree
#pragma unroll
    for (int cc = 0; cc < NCB; ++cc)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        for (int off = G; off < 32; off <<= 1) acc[cc][j] += __shfl_xor_sync(0xffffffffu, acc[cc][j], off);
    if (sub == 0) adagrad_row<TW, NCB>(t, e0, D, G, li, acc, lr, eps);
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

static size_t scatter_smem() {
  return sizeof(unsigned) * ((size_t)kSortWarps * kDigits + 2 * kDigits + 33 + 2 * (size_t)kSortTile);
}

template <typename TW, int G, int NCB>
static cudaError_t launch_reduce(const emb_table* t, const unsigned* K, const unsigned* V, const float* scale,
                                 int mean, const float* grad, unsigned n, unsigned n_bags, const WsLayout& L, char* ws,
                                 float lr, float eps, cudaStream_t st) {
  constexpr int U = NCB >= 4 ? 2 : 4;
  TableView v = t->view();
  const int threads = 256;
  long long blocks = ((long long)L.n_chunks * 32 + threads - 1) / threads;
  blocks = std::min<long long>(blocks, resident_blocks(threads));
  float* pa = (float*)(ws + L.partA);
  float* pb = (float*)(ws + L.partB);
  unsigned* ar = (unsigned*)(ws + L.arow);
  segreduce_adagrad_kernel<TW, G, NCB, U><<<(int)std::max(1LL, blocks), threads, 0, st>>>(
      v, K, V, scale, mean, grad, n, n_bags, L.n_chunks, pa, pb, ar, lr, eps);
  fixup_kernel<TW, G, NCB><<<(int)std::max(1LL, blocks), threads, 0, st>>>(v, K, n, L.n_chunks, pa, pb, ar, lr, eps);
  return cudaGetLastError();
}

template <typename TW>
static cudaError_t dispatch_reduce(const emb_table* t, const unsigned* K, const unsigned* V, const float* scale,
                                   int mean, const float* grad, unsigned n, unsigned n_bags, const WsLayout& L,
                                   char* ws, float lr, float eps, cudaStream_t st) {
  const int vecs = t->st.max_dim / 4;  // float4 columns of the widest row
  if (vecs <= 1) return launch_reduce<TW, 1, 1>(t, K, V, scale, mean, grad, n, n_bags, L, ws, lr, eps, st);
  if (vecs <= 2) return launch_reduce<TW, 2, 1>(t, K, V, scale, mean, grad, n, n_bags, L, ws, lr, eps, st);
  if (vecs <= 4) return launch_reduce<TW, 4, 1>(t, K, V, scale, mean, grad, n, n_bags, L, ws, lr, eps, st);
  if (vecs <= 8) return launch_reduce<TW, 8, 1>(t, K, V, scale, mean, grad, n, n_bags, L, ws, lr, eps, st);
  if (vecs <= 16) return launch_reduce<TW, 8, 2>(t, K, V, scale, mean, grad, n, n_bags, L, ws, lr, eps, st);
  if (vecs <= 32) return launch_reduce<TW, 8, 4>(t, K, V, scale, mean, grad, n, n_bags, L, ws, lr, eps, st);
  if (vecs <= 64) return launch_reduce<TW, 8, 8>(t, K, V, scale, mean, grad, n, n_bags, L, ws, lr, eps, st);
  return launch_reduce<TW, 8, 16>(t, K, V, scale, mean, grad, n, n_bags, L, ws, lr, eps, st);
}

static int bits_for(unsigned x) {
  int b = 0;
  while (b < 32 && (x >> b) != 0) ++b;
  return b;
}

static emb_status run_bwd(emb_table* table, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                          int64_t nnz, emb_pool pool, const float* grad_out_d, float lr, float eps, char* ws,
                          const WsLayout& L, cudaStream_t st) {
  const unsigned n = (unsigned)nnz;
  const unsigned miss = (unsigned)table->st.n_keys;
  const int bits = bits_for(miss);  // rows and the miss sentinel fit in `bits`
  const int passes = std::max(1, (bits + kRadixBits - 1) / kRadixBits);
  const unsigned sorted_in_b = (unsigned)(passes & 1);
  TableView v = table->view();
  WsHeader* hdr = (WsHeader*)(ws + L.hdr);
  unsigned* kA = (unsigned*)(ws + L.kA);
  unsigned* kB = (unsigned*)(ws + L.kB);
  unsigned* vA = (unsigned*)(ws + L.vA);
  unsigned* vB = (unsigned*)(ws + L.vB);
  float* scale = (float*)(ws + L.scale);
  const int mean = pool == EMB_POOL_MEAN;

  // With malformed offsets (flagged) some positions keep stale values; every
  // later kernel treats rows >= n_rows and bags >= n_bags as absent, so they
  // stay in bounds.
  long long blocks = std::min<long long>((n_bags * 32 + 255) / 256, resident_blocks(256));
  expand_kernel<<<(int)std::max(1LL, blocks), 256, 0, st>>>(v, (const long long*)offsets_d, n_bags,
                                                            (const long long*)keys_d, nnz, mean, kA, vA, scale, hdr,
                                                            sorted_in_b);
  EMB_CUDA(cudaGetLastError());
  if (nnz == 0) return EMB_OK;

  unsigned* counts = (unsigned*)(ws + L.counts);
  unsigned* partials = (unsigned*)(ws + L.partials);
  const size_t smem = scatter_smem();
  EMB_CUDA(cudaFuncSetAttribute(radix_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  unsigned *ki = kA, *vi = vA, *ko = kB, *vo = vB;
  for (int p = 0; p < passes; ++p) {
    const int shift = p * kRadixBits;
    radix_count_kernel<<<L.n_tiles_sort, kSortThreads, 0, st>>>(ki, n, shift, counts, L.n_tiles_sort);
    EMB_CUDA(launch_scan(counts, counts, (size_t)kDigits * L.n_tiles_sort, partials, st));
    radix_scatter_kernel<<<L.n_tiles_sort, kSortThreads, smem, st>>>(ki, vi, ko, vo, n, shift, counts,
                                                                     L.n_tiles_sort);
    EMB_CUDA(cudaGetLastError());
    std::swap(ki, ko);
    std::swap(vi, vo);
  }
  // ki/vi hold the sorted pairs
  cudaError_t e = table->st.wdtype == EMB_F16
                      ? dispatch_reduce<__half>(table, ki, vi, scale, mean, grad_out_d, n, (unsigned)n_bags, L, ws, lr, eps, st)
                      : dispatch_reduce<float>(table, ki, vi, scale, mean, grad_out_d, n, (unsigned)n_bags, L, ws, lr, eps, st);
  if (e != cudaSuccess) return cuda_fail(e, "segmented reduce launch");
  return EMB_OK;
}

// Scratch for emb_bwd_adagrad_noalloc, for callers that cannot allocate
// device memory.  The loader reserves it on every GPU that loads this library;
// host code must not pass the symbol itself to a kernel (on the host it only
// names a stand-in), so each device's address is looked up once.
static __device__ __align__(256) unsigned char g_noalloc_scratch[EMB_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[kMaxDevices] = {};

static emb_status noalloc_scratch(void** out) {
  int dev = 0;
  EMB_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return fail(EMB_ERR_UNSUPPORTED, "device index beyond the no-alloc table");
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
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
  if (n_bags > 0 && !grad_out_d) return fail(EMB_ERR_INVALID_ARG, "grad_out is NULL");
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
  return run_bwd(table, offsets_d, n_bags, keys_d, nnz, pool, grad_out_d, lr, eps, (char*)scratch, L,
                 (cudaStream_t)stream);
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
  emb_status rc = check_batch(table, offsets_d, n_bags, keys_d, nnz, pool);
  if (rc != EMB_OK) return rc;
  if (n_bags > 0 && !grad_out_d) return fail(EMB_ERR_INVALID_ARG, "grad_out is NULL");
  const WsLayout L = ws_layout(table, n_bags, nnz);
  if (!workspace_d || ws_bytes < L.total) return fail(EMB_ERR_WORKSPACE, "workspace missing or too small");
  if (((uintptr_t)workspace_d & 255) != 0) return fail(EMB_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  return run_bwd(table, offsets_d, n_bags, keys_d, nnz, pool, grad_out_d, lr, eps, (char*)workspace_d, L,
                 (cudaStream_t)stream);
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
