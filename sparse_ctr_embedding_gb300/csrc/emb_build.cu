// Device-side table build: emb_table_create_device.
//
// The Tencent PCG DataFun talk ("各阶段优化详细介绍") prepares the
// insert-free table before a pass and flashes it to GPU memory whole.  This
// file prepares it on the GPU from keys already in device memory, and
// reproduces exactly the layout of the host preparation (emb_table_create):
// keys inserted one by one in keys-array order, each into the first free
// slot at or after fmix64(key) mod capacity (linear probing, wrapping), rows
// renumbered slot-major, stable in keys-array order.
//
// How the sequential insertion is reproduced in parallel:
//  1. The set of occupied slots does not depend on the insertion order.  With
//     the keys sorted by home (stable), inserting them in that order puts the
//     j-th at p_j = max(h_j, p_{j-1} + 1) = j + max_{i<=j} (h_i - i): a
//     prefix-max scan.  Positions past the end spill over to the start.
//  2. If anything spills, the (o+1)-th empty slot of that unwrapped layout (o
//     the spill) stays empty once the spill is wrapped, so the circle is cut
//     just after it: homes are rotated to start there and the scan repeated,
//     which then spills nothing.
//  3. In that frame every maximal run of consecutive positions holds exactly
//     the keys whose homes lie in it, and no key of a run is ever pushed out
//     of it, whatever the order: runs are independent.  One warp (one block
//     for a run longer than 256 keys) replays its run's insertions in
//     keys-array order with an occupancy bitmask, which gives every key its
//     slot, its probe length and, on the way, duplicate keys.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <vector>

#include "emb_internal.cuh"

namespace emb {

constexpr int kWarpRun = 256;   // runs up to this length are replayed by one warp
constexpr int kMaxRun = 4096;   // longer runs are refused (EMB_ERR_UNSUPPORTED)
constexpr int kMaxScanThreads = 256;
constexpr int kMaxScanItems = 8;
constexpr int kMaxScanTile = kMaxScanThreads * kMaxScanItems;
constexpr long long kNegInf = -(1LL << 62);

struct BuildInfo {
  unsigned long long min_reserved;  // smallest keys-array index holding the reserved key -1
  unsigned long long min_badslot;   // smallest index whose slot field is >= n_slots
  unsigned long long min_dup;       // smallest index whose key equals a key earlier in the array
  unsigned long long sum_probe;
  unsigned long long max_probe;
  unsigned long long max_run;
  unsigned long long n_long;        // runs longer than kWarpRun, listed for the block replay
  unsigned long long too_long;      // a run longer than kMaxRun
  unsigned long long bad;           // a replay found no free slot in its run (never on a valid layout)
  unsigned long long r0;            // the rotated frame starts at slot r0
  unsigned long long rot;           // first index (in home order) of a key whose home is >= r0
  long long merged;                 // first + last run, if they touch across the end of the table
};

// ------------------------------------------------------------------ homes, validation, slot counts

__global__ void __launch_bounds__(256) build_home_kernel(const long long* __restrict__ keys, unsigned n,
                                                         unsigned long long mask, unsigned n_slots,
                                                         unsigned* __restrict__ H, unsigned* __restrict__ I,
                                                         unsigned* __restrict__ slotf,
                                                         unsigned* __restrict__ slot_count, BuildInfo* info) {
  extern __shared__ unsigned hist[];  // per-block slot histogram when n_slots is small (else unused)
  const bool local = n_slots <= 4096;
  if (local)
    for (unsigned s = threadIdx.x; s < n_slots; s += blockDim.x) hist[s] = 0;
  __syncthreads();
  for (unsigned i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const long long k = keys[i];
    const unsigned s = (unsigned)key_slot(k);
    if (k == kEmptyKey) {
      atomicMin(&info->min_reserved, (unsigned long long)i);
    } else if (s >= n_slots) {
      atomicMin(&info->min_badslot, (unsigned long long)i);
    } else if (local) {
      atomicAdd(&hist[s], 1u);
    } else {
      atomicAdd(&slot_count[s], 1u);
    }
    H[i] = (unsigned)(fmix64((unsigned long long)k) & mask);
    I[i] = i;
    slotf[i] = s < n_slots ? s : 0u;
  }
  __syncthreads();
  if (local)
    for (unsigned s = threadIdx.x; s < n_slots; s += blockDim.x)
      if (hist[s]) atomicAdd(&slot_count[s], hist[s]);
}

__global__ void iota_kernel(unsigned* __restrict__ v, unsigned n) {
  for (unsigned i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) v[i] = i;
}

// ------------------------------------------------------------------ prefix-max scan of h_j - j

__device__ __forceinline__ long long block_excl_max(long long v, long long* sm) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int nw = (int)(blockDim.x >> 5);
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = max(x, y);
  }
  __syncthreads();
  if (lane == 31) sm[w] = x;
  __syncthreads();
  if (w == 0) {
    const long long t = lane < nw ? sm[lane] : kNegInf;
    long long incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl = max(incl, y);
    }
    const long long ex = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane < nw) sm[lane] = lane == 0 ? kNegInf : ex;
    if (lane == nw - 1) sm[32] = incl;
  }
  __syncthreads();
  const long long before_warp = sm[w];
  const long long before_lane = __shfl_up_sync(0xffffffffu, x, 1);
  return max(before_warp, lane == 0 ? kNegInf : before_lane);
}

__global__ void __launch_bounds__(kMaxScanThreads) maxscan_reduce_kernel(const unsigned* __restrict__ h, unsigned n,
                                                                         long long* __restrict__ part) {
  __shared__ long long sm[33];
  const unsigned base = blockIdx.x * kMaxScanTile;
  long long m = kNegInf;
#pragma unroll
  for (int j = 0; j < kMaxScanItems; ++j) {
    const unsigned i = base + j * kMaxScanThreads + threadIdx.x;
    if (i < n) m = max(m, (long long)h[i] - (long long)i);
  }
  block_excl_max(m, sm);
  if (threadIdx.x == 0) part[blockIdx.x] = sm[32];
}

// one block: exclusive prefix max of the tile maxima, in place
__global__ void __launch_bounds__(1024) maxscan_partials_kernel(long long* part, unsigned np) {
  __shared__ long long sm[33];
  __shared__ long long carry;
  if (threadIdx.x == 0) carry = kNegInf;
  __syncthreads();
  for (unsigned b0 = 0; b0 < np; b0 += blockDim.x) {
    const unsigned i = b0 + threadIdx.x;
    const long long v = i < np ? part[i] : kNegInf;
    const long long ex = max(block_excl_max(v, sm), carry);
    const long long tot = sm[32];
    __syncthreads();
    if (i < np) part[i] = ex;
    if (threadIdx.x == 0) carry = max(carry, tot);
    __syncthreads();
  }
}

// p_j = j + max_{i <= j} (h_i - i)
__global__ void __launch_bounds__(kMaxScanThreads) maxscan_down_kernel(const unsigned* __restrict__ h, unsigned n,
                                                                       const long long* __restrict__ part,
                                                                       long long* __restrict__ P) {
  __shared__ long long sm[33];
  const unsigned base = blockIdx.x * kMaxScanTile + threadIdx.x * kMaxScanItems;
  long long v[kMaxScanItems];
  long long m = kNegInf;
#pragma unroll
  for (int j = 0; j < kMaxScanItems; ++j) {
    const unsigned i = base + j;
    v[j] = i < n ? (long long)h[i] - (long long)i : kNegInf;
    m = max(m, v[j]);
  }
  long long run = max(block_excl_max(m, sm), part[blockIdx.x]);
#pragma unroll
  for (int j = 0; j < kMaxScanItems; ++j) {
    const unsigned i = base + j;
    run = max(run, v[j]);
    if (i < n) P[i] = (long long)i + run;
  }
}

static cudaError_t launch_maxscan(const unsigned* h, unsigned n, long long* part, long long* P, cudaStream_t st) {
  const unsigned np = (n + kMaxScanTile - 1) / kMaxScanTile;
  maxscan_reduce_kernel<<<np, kMaxScanThreads, 0, st>>>(h, n, part);
  maxscan_partials_kernel<<<1, 1024, 0, st>>>(part, np);
  maxscan_down_kernel<<<np, kMaxScanThreads, 0, st>>>(h, n, part, P);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ the cut of the circle

// One thread.  spill o = p_{n-1} - (cap - 1).  If o > 0, the (o+1)-th empty
// slot e of the unwrapped layout (empties before p_j: p_j - j, nondecreasing)
// is cut after: r0 = e + 1; rot = first index in home order with h >= r0.
__global__ void plan_cut_kernel(const unsigned* __restrict__ SH, const long long* __restrict__ P, unsigned n,
                                unsigned long long cap, BuildInfo* info) {
  const long long o = P[n - 1] - (long long)(cap - 1);
  unsigned long long r0 = 0;
  if (o > 0) {
    unsigned lo = 0, hi = n - 1;  // smallest j with P_j - j >= o + 1 (exists: n <= cap / 2)
    while (lo < hi) {
      const unsigned mid = (lo + hi) >> 1;
      if (P[mid] - (long long)mid >= o + 1) hi = mid; else lo = mid + 1;
    }
    const long long e = lo == 0 ? o : P[lo - 1] + (o + 1 - (P[lo - 1] - (long long)(lo - 1)));
    r0 = (unsigned long long)(e + 1) & (cap - 1);
  }
  unsigned lo = 0, hi = n;  // first j with SH_j >= r0
  while (lo < hi) {
    const unsigned mid = (lo + hi) >> 1;
    if ((unsigned long long)SH[mid] >= r0) hi = mid; else lo = mid + 1;
  }
  info->r0 = r0;
  info->rot = r0 == 0 ? 0 : lo;
}

__global__ void rotate_kernel(const unsigned* __restrict__ SH, const unsigned* __restrict__ SI, unsigned n,
                              unsigned long long mask, const BuildInfo* __restrict__ info, unsigned* __restrict__ RH,
                              unsigned* __restrict__ RI) {
  const unsigned rot = (unsigned)info->rot;
  const unsigned long long r0 = info->r0;
  for (unsigned j2 = blockIdx.x * blockDim.x + threadIdx.x; j2 < n; j2 += gridDim.x * blockDim.x) {
    unsigned j = j2 + rot;
    if (j >= n) j -= n;
    RH[j2] = (unsigned)(((unsigned long long)SH[j] - r0) & mask);
    RI[j2] = SI[j];
  }
}

// ------------------------------------------------------------------ runs

__global__ void run_flag_kernel(const long long* __restrict__ P, unsigned n, unsigned* __restrict__ F) {
  for (unsigned j = blockIdx.x * blockDim.x + threadIdx.x; j < n; j += gridDim.x * blockDim.x)
    F[j] = (j == 0 || P[j] != P[j - 1] + 1) ? 1u : 0u;
}

__global__ void run_start_kernel(const unsigned* __restrict__ F, const unsigned* __restrict__ Fx, unsigned n,
                                 unsigned* __restrict__ RS) {
  for (unsigned j = blockIdx.x * blockDim.x + threadIdx.x; j < n; j += gridDim.x * blockDim.x)
    if (F[j]) RS[Fx[j]] = j;
}

// Replay of one run [a, a + m) by a group of threads (a warp, or a block for
// long runs), all of whose keys have rotated homes in [pa, pa + m):
// (1) load relative homes, indices and keys; (2) each key's rank by keys-array
// index (and duplicate pairs); (3) one thread inserts them in rank order into
// the run's occupancy bitmask.
template <int CAP>
struct RunSmem {
  unsigned hr[CAP];
  unsigned idx[CAP];
  long long key[CAP];
  unsigned short order[CAP];
  unsigned occ[(CAP + 31) / 32];
};

// The leader adds the run's probe lengths to *sum and raises *mx (its own
// running totals: one atomic per warp or block at the end, not per run).
template <int CAP>
__device__ void replay_run(RunSmem<CAP>& sm, const long long* __restrict__ keys, const unsigned* __restrict__ RH,
                           const unsigned* __restrict__ RI, const long long* __restrict__ P, unsigned a, unsigned m,
                           unsigned long long mask, unsigned long long r0, unsigned* __restrict__ fin,
                           BuildInfo* info, int tid, int nthreads, bool leader, unsigned long long* sum,
                           unsigned long long* mx) {
  const long long pa = P[a];
  for (unsigned t = tid; t < m; t += nthreads) {
    sm.hr[t] = (unsigned)((long long)RH[a + t] - pa);
    sm.idx[t] = RI[a + t];
    sm.key[t] = keys[sm.idx[t]];
  }
  for (unsigned w = tid; w < (m + 31) / 32; w += nthreads) sm.occ[w] = 0u;
  if (nthreads == 32) __syncwarp(); else __syncthreads();
  for (unsigned t = tid; t < m; t += nthreads) {
    const unsigned it = sm.idx[t];
    const long long kt = sm.key[t];
    unsigned r = 0;
    unsigned long long dup = ~0ULL;
    for (unsigned u = 0; u < m; ++u) {
      const unsigned iu = sm.idx[u];
      r += iu < it;
      if (u != t && sm.key[u] == kt) dup = min(dup, (unsigned long long)max(iu, it));
    }
    sm.order[r] = (unsigned short)t;
    if (dup != ~0ULL) atomicMin(&info->min_dup, dup);
  }
  if (nthreads == 32) __syncwarp(); else __syncthreads();
  if (leader) {
    const unsigned nw = (m + 31) / 32;
    for (unsigned q = 0; q < m; ++q) {
      const unsigned t = sm.order[q];
      const unsigned h = sm.hr[t];
      unsigned w = h >> 5;
      unsigned bits = w < nw ? (~sm.occ[w] & (0xFFFFFFFFu << (h & 31))) : 0u;
      while (!bits && ++w < nw) bits = ~sm.occ[w];
      const unsigned pos = w * 32 + (unsigned)(__ffs(bits) - 1);
      if (w >= nw || pos >= m) {  // cannot happen on a consistent run; report, do not write
        atomicOr(&info->bad, 1ULL);
        break;
      }
      sm.occ[w] |= 1u << (pos & 31);
      fin[sm.idx[t]] = (unsigned)(((unsigned long long)(pa + pos) + r0) & mask);
      const unsigned long long len = (unsigned long long)(pos - h + 1);
      *sum += len;
      *mx = max(*mx, len);
    }
  }
}

constexpr int kRunWarps = 4;

__global__ void __launch_bounds__(kRunWarps * 32) run_warp_kernel(
    const long long* __restrict__ keys, const unsigned* __restrict__ RH, const unsigned* __restrict__ RI,
    const long long* __restrict__ P, const unsigned* __restrict__ RS, const unsigned* __restrict__ n_runs_p, unsigned n,
    unsigned long long mask, const BuildInfo* __restrict__ cinfo, BuildInfo* info, unsigned* __restrict__ fin,
    unsigned* __restrict__ long_list) {
  __shared__ RunSmem<kWarpRun> sm[kRunWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned R = *n_runs_p;
  const unsigned long long r0 = cinfo->r0;
  const unsigned nwarps = gridDim.x * kRunWarps;
  unsigned long long sum = 0, mx = 0, mrun = 0;
  for (unsigned k = blockIdx.x * kRunWarps + w; k < R; k += nwarps) {
    const unsigned a = RS[k], b = k + 1 < R ? RS[k + 1] : n;
    const unsigned m = b - a;
    mrun = max(mrun, (unsigned long long)m);
    if (m > kWarpRun) {
      if (lane == 0) {
        if (m > kMaxRun) atomicOr(&info->too_long, 1ULL);
        else long_list[atomicAdd(&info->n_long, 1ULL)] = k;
      }
      continue;
    }
    replay_run<kWarpRun>(sm[w], keys, RH, RI, P, a, m, mask, r0, fin, info, lane, 32, lane == 0, &sum, &mx);
    __syncwarp();
  }
  if (lane == 0) {
    if (sum) atomicAdd(&info->sum_probe, sum);
    if (mx) atomicMax(&info->max_probe, mx);
    if (mrun) atomicMax(&info->max_run, mrun);
  }
}

__global__ void __launch_bounds__(256) run_block_kernel(
    const long long* __restrict__ keys, const unsigned* __restrict__ RH, const unsigned* __restrict__ RI,
    const long long* __restrict__ P, const unsigned* __restrict__ RS, const unsigned* __restrict__ n_runs_p, unsigned n,
    unsigned long long mask, const BuildInfo* __restrict__ cinfo, BuildInfo* info, unsigned* __restrict__ fin,
    const unsigned* __restrict__ long_list) {
  extern __shared__ __align__(16) unsigned char dyn[];
  RunSmem<kMaxRun>& sm = *reinterpret_cast<RunSmem<kMaxRun>*>(dyn);
  const unsigned R = *n_runs_p;
  const unsigned L = (unsigned)cinfo->n_long;
  const unsigned long long r0 = cinfo->r0;
  unsigned long long sum = 0, mx = 0;
  for (unsigned q = blockIdx.x; q < L; q += gridDim.x) {
    const unsigned k = long_list[q];
    const unsigned a = RS[k], b = k + 1 < R ? RS[k + 1] : n;
    replay_run<kMaxRun>(sm, keys, RH, RI, P, a, b - a, mask, r0, fin, info, threadIdx.x, blockDim.x,
                        threadIdx.x == 0, &sum, &mx);
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (sum) atomicAdd(&info->sum_probe, sum);
    if (mx) atomicMax(&info->max_probe, mx);
  }
}

// One thread: the first and last runs of the frame touch across the end of
// the table only when no cut was made and slots 0 and cap - 1 are both
// occupied; the longest cluster is then possibly their sum.
__global__ void merged_run_kernel(const long long* __restrict__ P, const unsigned* __restrict__ RS,
                                  const unsigned* __restrict__ n_runs_p, unsigned n, unsigned long long cap,
                                  BuildInfo* info) {
  const unsigned R = *n_runs_p;
  info->merged = 0;
  if (info->r0 == 0 && R > 1 && P[0] == 0 && P[n - 1] == (long long)(cap - 1))
    info->merged = (long long)(RS[1] - RS[0]) + (long long)(n - RS[R - 1]);
}

// ------------------------------------------------------------------ rows and slots

__global__ void row_maps_kernel(const long long* __restrict__ keys, const unsigned* __restrict__ int_to_ext,
                                unsigned n, unsigned* __restrict__ ext_to_int, long long* __restrict__ row_key) {
  for (unsigned r = blockIdx.x * blockDim.x + threadIdx.x; r < n; r += gridDim.x * blockDim.x) {
    const unsigned i = int_to_ext[r];
    ext_to_int[i] = r;
    row_key[r] = keys[i];
  }
}

__global__ void empty_slots_kernel(Slot* __restrict__ slots, unsigned long long cap) {
  for (unsigned long long p = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; p < cap;
       p += (unsigned long long)gridDim.x * blockDim.x)
    slots[p] = Slot{kEmptyKey, 0u, 0u};
}

__global__ void place_slots_kernel(const long long* __restrict__ keys, const unsigned* __restrict__ fin,
                                   const unsigned* __restrict__ ext_to_int, unsigned n, Slot* __restrict__ slots) {
  for (unsigned i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    slots[fin[i]] = Slot{keys[i], ext_to_int[i], i};
}

static int grid_of(unsigned long long work) {
  const unsigned long long g = (work + 255) / 256;
  return (int)std::max<unsigned long long>(1, std::min<unsigned long long>(g, (unsigned long long)sm_count() * 16));
}

static int bits_of(unsigned long long x) {
  int b = 0;
  while (b < 64 && (x >> b) != 0) ++b;
  return b;
}

}  // namespace emb

using namespace emb;

extern "C" emb_status emb_table_create_device(const emb_table_desc* desc, const int64_t* keys_d, int64_t n_keys,
                                              const void* values, const float* acc, void* stream, emb_table** out) {
  if (!out) return fail(EMB_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  int64_t cap = 0;
  int max_dim = 0;
  long long sum_dims = 0;
  emb_status rc = check_desc(desc, n_keys, &cap, &max_dim, &sum_dims);
  if (rc != EMB_OK) return rc;
  if (n_keys > 0 && !keys_d) return fail(EMB_ERR_INVALID_ARG, "keys is NULL");
  if (cap > (1LL << 32)) return fail(EMB_ERR_UNSUPPORTED, "the device build takes capacities up to 2^32");
  const unsigned n = (unsigned)n_keys;
  const unsigned long long mask = (unsigned long long)cap - 1;
  const unsigned S = (unsigned)desc->n_slots;
  cudaStream_t st = (cudaStream_t)stream;
  const long long* keys = (const long long*)keys_d;

  emb_table* t = new (std::nothrow) emb_table();
  if (!t) return fail(EMB_ERR_OOM, "host allocation failed");
  cudaGetDevice(&t->device);
  t->optimizer = (int)desc->optimizer;

  // scratch (freed before return)
  std::vector<void*> scratch;
  auto salloc = [&](void** p, size_t bytes) -> cudaError_t {
    cudaError_t e = dmalloc(p, std::max<size_t>(bytes, 16));
    if (e == cudaSuccess) scratch.push_back(*p);
    return e;
  };
  uint64_t bytes = 0;
  auto body = [&]() -> emb_status {
    const size_t nn = std::max<unsigned>(n, 1);
    unsigned *H0, *I0, *H1, *I1, *slotf, *F, *Fx, *RS, *fin, *cnt, *part32, *long_list;
    long long *P, *part64;
    BuildInfo* info;
    void* sortscr;
    const unsigned np64 = (n + kMaxScanTile - 1) / kMaxScanTile + 1;
    const size_t np32 = (nn + 4095) / 4096 + 2;
    EMB_CUDA(salloc((void**)&H0, nn * 4));
    EMB_CUDA(salloc((void**)&I0, nn * 4));
    EMB_CUDA(salloc((void**)&H1, nn * 4));
    EMB_CUDA(salloc((void**)&I1, nn * 4));
    EMB_CUDA(salloc((void**)&slotf, nn * 4));
    EMB_CUDA(salloc((void**)&F, nn * 4));
    EMB_CUDA(salloc((void**)&Fx, nn * 4));
    EMB_CUDA(salloc((void**)&RS, nn * 4));
    EMB_CUDA(salloc((void**)&fin, nn * 4));
    EMB_CUDA(salloc((void**)&long_list, nn * 4));
    EMB_CUDA(salloc((void**)&cnt, (size_t)S * 4));
    EMB_CUDA(salloc((void**)&part32, np32 * 4));
    EMB_CUDA(salloc((void**)&P, nn * 8));
    EMB_CUDA(salloc((void**)&part64, (size_t)np64 * 8));
    EMB_CUDA(salloc((void**)&info, sizeof(BuildInfo)));
    EMB_CUDA(salloc(&sortscr, pair_sort_scratch_bytes((unsigned)nn)));

    BuildInfo init{};
    init.min_reserved = init.min_badslot = init.min_dup = ~0ULL;
    EMB_CUDA(cudaMemcpyAsync(info, &init, sizeof init, cudaMemcpyHostToDevice, st));
    EMB_CUDA(cudaMemsetAsync(cnt, 0, (size_t)S * 4, st));
    if (n > 0) {
      build_home_kernel<<<grid_of(n), 256, S <= 4096 ? S * 4 : 0, st>>>(keys, n, mask, S, H0, I0, slotf, cnt, info);
      EMB_CUDA(cudaGetLastError());
    }
    BuildInfo hi{};
    std::vector<unsigned> counts(S);
    EMB_CUDA(cudaMemcpyAsync(&hi, info, sizeof hi, cudaMemcpyDeviceToHost, st));
    EMB_CUDA(cudaMemcpyAsync(counts.data(), cnt, (size_t)S * 4, cudaMemcpyDeviceToHost, st));
    EMB_CUDA(cudaStreamSynchronize(st));
    if (hi.min_reserved != ~0ULL || hi.min_badslot != ~0ULL) {
      char buf[128];
      if (hi.min_reserved <= hi.min_badslot) return fail(EMB_ERR_RESERVED_KEY, "key -1 is the empty-slot sentinel");
      std::snprintf(buf, sizeof buf, "key index %llu has slot field >= n_slots", hi.min_badslot);
      return fail(EMB_ERR_INVALID_ARG, buf);
    }

    // the slot layout
    if (n > 0) {
      bool in_b = false;
      EMB_CUDA(pair_sort(H0, I0, H1, I1, n, bits_of(mask), sortscr, st, &in_b));
      const unsigned* SH = in_b ? H1 : H0;
      const unsigned* SI = in_b ? I1 : I0;
      unsigned* RH = in_b ? H0 : H1;  // the other pair of buffers takes the rotated frame
      unsigned* RI = in_b ? I0 : I1;
      EMB_CUDA(launch_maxscan(SH, n, part64, P, st));
      plan_cut_kernel<<<1, 1, 0, st>>>(SH, P, n, (unsigned long long)cap, info);
      rotate_kernel<<<grid_of(n), 256, 0, st>>>(SH, SI, n, mask, info, RH, RI);
      EMB_CUDA(launch_maxscan(RH, n, part64, P, st));
      run_flag_kernel<<<grid_of(n), 256, 0, st>>>(P, n, F);
      EMB_CUDA(launch_scan_u32(F, Fx, n, part32, st));
      const unsigned np = (n + 4095) / 4096;  // the scan's tile count: its total lands in part32[np]
      run_start_kernel<<<grid_of(n), 256, 0, st>>>(F, Fx, n, RS);
      const unsigned* n_runs = part32 + np;
      run_warp_kernel<<<sm_count() * 8, kRunWarps * 32, 0, st>>>(keys, RH, RI, P, RS, n_runs, n, mask, info, info,
                                                                 fin, long_list);
      const int big = (int)sizeof(RunSmem<kMaxRun>);
      EMB_CUDA(cudaFuncSetAttribute(run_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, big));
      run_block_kernel<<<sm_count(), 256, big, st>>>(keys, RH, RI, P, RS, n_runs, n, mask, info, info, fin, long_list);
      merged_run_kernel<<<1, 1, 0, st>>>(P, RS, n_runs, n, (unsigned long long)cap, info);
      EMB_CUDA(cudaGetLastError());
      EMB_CUDA(cudaMemcpyAsync(&hi, info, sizeof hi, cudaMemcpyDeviceToHost, st));
      EMB_CUDA(cudaStreamSynchronize(st));
      if (hi.min_dup != ~0ULL) {
        char buf[96];
        std::snprintf(buf, sizeof buf, "duplicate key at keys-array index %llu", hi.min_dup);
        return fail(EMB_ERR_DUP_KEY, buf);
      }
      if (hi.too_long) return fail(EMB_ERR_UNSUPPORTED, "a run of occupied slots longer than the device build takes "
                                                        "(4096): use emb_table_create");
      if (hi.bad) return fail(EMB_ERR_CUDA, "device build: inconsistent run (internal error)");
    }

    // statistics and the slot-major row numbering (stable in keys-array order)
    emb_table_stats& s = t->st;
    std::memset(&s, 0, sizeof s);
    s.n_keys = n_keys;
    s.capacity = cap;
    s.n_slots = (int32_t)S;
    s.sum_dims = (int32_t)sum_dims;
    s.max_dim = max_dim;
    s.wdtype = (int32_t)desc->wdtype;
    s.load_factor = (double)n_keys / (double)cap;
    s.sum_probe = (int64_t)hi.sum_probe;
    s.max_probe = (int64_t)hi.max_probe;
    s.max_cluster = std::max<int64_t>((int64_t)hi.max_run, hi.merged);
    s.probe_bound = s.max_cluster + 1;
    t->sinfo_h.resize(S);
    long long row = 0, elem = 0, col = 0;
    for (unsigned q = 0; q < S; ++q) {
      SlotInfo& si = t->sinfo_h[q];
      si.dim = desc->slot_dim[q];
      si.col = (int)col;
      si.row_base = (unsigned)row;
      si.n_rows = counts[q];
      si.elem_base = elem;
      row += counts[q];
      elem += (long long)counts[q] * si.dim;
      col += si.dim;
      s.max_slot_keys = std::max<int64_t>(s.max_slot_keys, counts[q]);
    }
    s.n_elems = elem;
    const bool ragged = std::any_of(desc->slot_dim, desc->slot_dim + S, [&](int x) { return x != desc->slot_dim[0]; });
    t->uniform_dim = ragged ? 0 : desc->slot_dim[0];

    auto talloc = [&](void** p, size_t b) -> cudaError_t {
      cudaError_t e = dmalloc(p, std::max<size_t>(b, 1));
      if (e == cudaSuccess) bytes += std::max<size_t>(b, 1);
      return e;
    };
    EMB_CUDA(talloc((void**)&t->slots_d, (size_t)cap * sizeof(Slot)));
    EMB_CUDA(talloc((void**)&t->sinfo_d, (size_t)S * sizeof(SlotInfo)));
    EMB_CUDA(talloc((void**)&t->row_key_d, nn * 8));
    EMB_CUDA(talloc((void**)&t->int_to_ext_d, nn * 4));
    EMB_CUDA(talloc((void**)&t->ext_to_int_d, nn * 4));
    EMB_CUDA(cudaMemcpyAsync(t->sinfo_d, t->sinfo_h.data(), (size_t)S * sizeof(SlotInfo), cudaMemcpyHostToDevice, st));
    empty_slots_kernel<<<grid_of((unsigned long long)cap), 256, 0, st>>>(t->slots_d, (unsigned long long)cap);
    if (n > 0) {
      iota_kernel<<<grid_of(n), 256, 0, st>>>(I0, n);
      bool in_b = false;
      EMB_CUDA(pair_sort(slotf, I0, H1, I1, n, std::max(1, bits_of(S - 1)), sortscr, st, &in_b));
      EMB_CUDA(cudaMemcpyAsync(t->int_to_ext_d, in_b ? I1 : I0, (size_t)n * 4, cudaMemcpyDeviceToDevice, st));
      row_maps_kernel<<<grid_of(n), 256, 0, st>>>(keys, t->int_to_ext_d, n, t->ext_to_int_d, t->row_key_d);
      place_slots_kernel<<<grid_of(n), 256, 0, st>>>(keys, fin, t->ext_to_int_d, n, t->slots_d);
      EMB_CUDA(cudaGetLastError());
    }
    if (ragged && n > 0) {  // element offsets of keys-array rows: prefix over the keys' dims (host)
      std::vector<long long> kh(n);
      EMB_CUDA(cudaMemcpyAsync(kh.data(), keys, (size_t)n * 8, cudaMemcpyDeviceToHost, st));
      EMB_CUDA(cudaStreamSynchronize(st));
      t->ext_elem_off_h.resize((size_t)n + 1);
      t->ext_elem_off_h[0] = 0;
      for (unsigned i = 0; i < n; ++i)
        t->ext_elem_off_h[i + 1] = t->ext_elem_off_h[i] + desc->slot_dim[((unsigned long long)kh[i]) >> 48];
      EMB_CUDA(talloc((void**)&t->ext_elem_off_d, ((size_t)n + 1) * 8));
      EMB_CUDA(cudaMemcpyAsync(t->ext_elem_off_d, t->ext_elem_off_h.data(), ((size_t)n + 1) * 8,
                               cudaMemcpyHostToDevice, st));
    }
    EMB_CUDA(cudaStreamSynchronize(st));
    return finish_table(t, desc, values, acc, st, &bytes);
  };
  rc = body();
  cudaStreamSynchronize(st);
  for (void* p : scratch) dfree(p);
  if (rc != EMB_OK) {
    free_table(t);
    return rc;
  }
  *out = t;
  return EMB_OK;
}
