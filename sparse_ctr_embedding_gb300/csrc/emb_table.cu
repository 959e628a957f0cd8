// Table preparation, upload, checkpoint export, probe-only resolve and the
// device flag.
//
// The table follows the insert-free GPU hashtable of the Tencent PCG DataFun
// talk ("各阶段优化详细介绍"): the whole structure is prepared on the host from
// the pass's deduplicated keys and copied to global memory in one block; the
// GPU never inserts.  Keys follow the unified layout of the same talk
// ("计算优化"): slot id in the high 16 bits, raw feature id in the low 48.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "emb_internal.cuh"

namespace emb {

// ------------------------------------------------------------------ errors

static thread_local std::string g_last_error;

emb_status fail(emb_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

emb_status cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  cudaGetLastError();  // clear a sticky launch error of this thread
  return e == cudaErrorMemoryAllocation ? EMB_ERR_OOM : EMB_ERR_CUDA;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

// ------------------------------------------------------------------ device allocations
//
// Every device allocation of the library goes through dmalloc/dfree, which
// count the live ones and can be told (emb_debug_fail_device_alloc) to fail
// from the N-th call on, so tests can check that a failed create returns
// EMB_ERR_OOM and leaves nothing allocated.

static std::atomic<long long> g_live_allocs{0};
static std::atomic<long long> g_fail_after{-1};  // < 0: never fail

cudaError_t dmalloc(void** p, size_t bytes) {
  long long left = g_fail_after.load();
  while (left >= 0) {
    if (left == 0) {
      *p = nullptr;
      return cudaErrorMemoryAllocation;
    }
    if (g_fail_after.compare_exchange_weak(left, left - 1)) break;
  }
  cudaError_t e = cudaMalloc(p, bytes);
  if (e == cudaSuccess) g_live_allocs.fetch_add(1);
  return e;
}

void dfree(void* p) {
  if (!p) return;
  cudaFree(p);
  g_live_allocs.fetch_sub(1);
}

static unsigned long long host_fmix64(unsigned long long k) {
  k ^= k >> 33;
  k *= 0xff51afd7ed558ccdULL;
  k ^= k >> 33;
  k *= 0xc4ceb9fe1a85ec53ULL;
  k ^= k >> 33;
  return k;
}

// ------------------------------------------------------------------ host plan

// Validate and prepare the table on the host.  Rows are renumbered
// slot-major (stable within a slot, i.e. in keys-array order); slots are
// filled by inserting keys one by one in keys-array order with linear
// probing, so the layout depends on that order alone.
// Validate a table description for n keys: dims, types and the capacity
// (0 = the smallest power of two >= 2 n).
emb_status check_desc(const emb_table_desc* d, int64_t n, int64_t* cap_out, int* max_dim_out,
                      long long* sum_dims_out) {
  if (!d) return fail(EMB_ERR_INVALID_ARG, "desc is NULL");
  if (n < 0) return fail(EMB_ERR_INVALID_ARG, "n_keys < 0");
  if (n > EMB_MAX_KEYS) return fail(EMB_ERR_UNSUPPORTED, "n_keys exceeds EMB_MAX_KEYS");
  if (d->n_slots < 1 || d->n_slots > 65535 || !d->slot_dim)
    return fail(EMB_ERR_INVALID_ARG, "n_slots must be in [1, 65535] with slot_dim given");
  if (d->wdtype != EMB_F32 && d->wdtype != EMB_F16 && d->wdtype != EMB_F16_MASTER)
    return fail(EMB_ERR_INVALID_ARG, "bad wdtype");
  if (d->optimizer != EMB_OPT_ADAGRAD && d->optimizer != EMB_OPT_FTRL && d->optimizer != EMB_OPT_ROWWISE_ADAGRAD)
    return fail(EMB_ERR_INVALID_ARG, "bad optimizer");
  const int vec = d->wdtype == EMB_F32 ? 4 : 8;
  int max_dim = 0;
  long long sum_dims = 0;
  for (int s = 0; s < d->n_slots; ++s) {
    int D = d->slot_dim[s];
    if (D < 1 || D > EMB_MAX_DIM) return fail(EMB_ERR_UNSUPPORTED, "slot dim outside [1, EMB_MAX_DIM]");
    if (D % vec) return fail(EMB_ERR_UNSUPPORTED, "slot dim must be a multiple of 4 (f32) or 8 (f16)");
    max_dim = std::max(max_dim, D);
    sum_dims += D;
  }
  if (sum_dims > (1LL << 30)) return fail(EMB_ERR_UNSUPPORTED, "sum of dims too large");
  int64_t cap = d->capacity;
  if (cap == 0) {
    cap = 2;
    while (cap < 2 * n) cap <<= 1;
  } else if (cap < 2 || (cap & (cap - 1)) != 0 || cap < 2 * n) {
    return fail(EMB_ERR_LOAD_FACTOR, "capacity must be a power of two >= 2 * n_keys");
  }
  if (cap > (1LL << 40)) return fail(EMB_ERR_UNSUPPORTED, "capacity too large");
  *cap_out = cap;
  *max_dim_out = max_dim;
  *sum_dims_out = sum_dims;
  return EMB_OK;
}

static emb_status build_plan(const emb_table_desc* d, const int64_t* keys, int64_t n, HostPlan& P,
                             bool with_slots) {
  int64_t cap = 0;
  int max_dim = 0;
  long long sum_dims = 0;
  emb_status rc0 = check_desc(d, n, &cap, &max_dim, &sum_dims);
  if (rc0 != EMB_OK) return rc0;
  if (n > 0 && !keys) return fail(EMB_ERR_INVALID_ARG, "keys is NULL");
  P.n_slots = d->n_slots;
  P.dims.assign(d->slot_dim, d->slot_dim + d->n_slots);
  P.wdtype = d->wdtype;
  P.n_keys = n;
  P.cap = cap;

  // per-slot counts, reserved and out-of-range keys
  std::vector<int64_t> count((size_t)P.n_slots, 0);
  for (int64_t i = 0; i < n; ++i) {
    if (keys[i] == kEmptyKey) return fail(EMB_ERR_RESERVED_KEY, "key -1 is the empty-slot sentinel");
    unsigned s = (unsigned)(((unsigned long long)keys[i]) >> 48);
    if ((int)s >= P.n_slots) {
      char buf[128];
      std::snprintf(buf, sizeof buf, "key index %lld has slot field %u >= n_slots", (long long)i, s);
      return fail(EMB_ERR_INVALID_ARG, buf);
    }
    count[s]++;
  }
  P.sinfo.resize((size_t)P.n_slots);
  long long row = 0, elem = 0, col = 0;
  for (int s = 0; s < P.n_slots; ++s) {
    SlotInfo& si = P.sinfo[(size_t)s];
    si.dim = P.dims[(size_t)s];
    si.col = (int)col;
    si.row_base = (unsigned)row;
    si.n_rows = (unsigned)count[(size_t)s];
    si.elem_base = elem;
    row += count[(size_t)s];
    elem += count[(size_t)s] * (long long)si.dim;
    col += si.dim;
  }
  const bool ragged = std::any_of(P.dims.begin(), P.dims.end(), [&](int x) { return x != P.dims[0]; });
  try {
    P.ext_to_int.resize((size_t)n);
    P.int_to_ext.resize((size_t)n);
    P.row_key.resize((size_t)n);
    std::vector<unsigned> cursor((size_t)P.n_slots);
    for (int s = 0; s < P.n_slots; ++s) cursor[(size_t)s] = P.sinfo[(size_t)s].row_base;
    for (int64_t i = 0; i < n; ++i) {
      unsigned s = (unsigned)(((unsigned long long)keys[i]) >> 48);
      unsigned r = cursor[s]++;
      P.ext_to_int[(size_t)i] = r;
      P.int_to_ext[r] = (uint32_t)i;
      P.row_key[r] = keys[i];
    }
    if (ragged) {
      P.ext_elem_off.resize((size_t)n + 1);
      P.ext_elem_off[0] = 0;
      for (int64_t i = 0; i < n; ++i)
        P.ext_elem_off[(size_t)i + 1] = P.ext_elem_off[(size_t)i] + P.dims[((unsigned long long)keys[i]) >> 48];
    }
  } catch (const std::bad_alloc&) {
    return fail(EMB_ERR_OOM, "host allocation failed while planning the table");
  }

  emb_table_stats& st = P.st;
  std::memset(&st, 0, sizeof st);
  st.n_keys = n;
  st.capacity = cap;
  st.n_elems = elem;
  st.n_slots = P.n_slots;
  st.sum_dims = (int32_t)sum_dims;
  st.max_dim = max_dim;
  st.wdtype = (int32_t)P.wdtype;
  st.load_factor = (double)n / (double)cap;
  for (int s = 0; s < P.n_slots; ++s) st.max_slot_keys = std::max<int64_t>(st.max_slot_keys, count[(size_t)s]);

  // sequential insertion in keys-array order; home slots of upcoming keys are
  // prefetched (a pure memory hint: the insertion order is unchanged)
  std::vector<Slot> local;
  std::vector<Slot>& slots = with_slots ? P.slots : local;
  try {
    slots.assign((size_t)cap, Slot{kEmptyKey, 0u, 0u});
  } catch (const std::bad_alloc&) {
    return fail(EMB_ERR_OOM, "host allocation of the slot array failed");
  }
  const unsigned long long mask = (unsigned long long)cap - 1;
  constexpr int64_t kAhead = 24;
  for (int64_t i = 0; i < n; ++i) {
    if (i + kAhead < n) __builtin_prefetch(&slots[host_fmix64((unsigned long long)keys[i + kAhead]) & mask], 1);
    const long long k = keys[i];
    unsigned long long h = host_fmix64((unsigned long long)k) & mask;
    int64_t len = 1;
    while (slots[h].key != kEmptyKey) {
      if (slots[h].key == k) {
        char buf[96];
        std::snprintf(buf, sizeof buf, "duplicate key at keys-array index %lld", (long long)i);
        return fail(EMB_ERR_DUP_KEY, buf);
      }
      h = (h + 1) & mask;
      ++len;
    }
    slots[h] = Slot{k, P.ext_to_int[(size_t)i], (unsigned)i};
    st.sum_probe += len;
    if (len > st.max_probe) st.max_probe = len;
  }
  // longest cyclic run of occupied slots (there is always an empty slot)
  if (n > 0) {
    unsigned long long e = 0;
    while (slots[e].key != kEmptyKey) ++e;
    int64_t run = 0;
    for (unsigned long long j = 1; j <= (unsigned long long)cap; ++j) {
      if (slots[(e + j) & mask].key != kEmptyKey) {
        if (++run > st.max_cluster) st.max_cluster = run;
      } else {
        run = 0;
      }
    }
  }
  st.probe_bound = st.max_cluster + 1;
  if (st.probe_bound > (1LL << 30)) return fail(EMB_ERR_UNSUPPORTED, "probe bound too large");
  return EMB_OK;
}

// ------------------------------------------------------------------ kernels

__device__ __forceinline__ long long ext_elem(const long long* ext_off, int uniform_dim, unsigned e) {
  return ext_off ? ext_off[e] : (long long)e * uniform_dim;
}

// Copy rows [e0, e1) of a keys-array-ordered ragged array (chunk base element
// src_base) into internal row order (to_int) or back (to_ext).  One warp per row.
template <typename T, bool kToInt>
__global__ void permute_rows_kernel(TableView t, const unsigned* ext_to_int, const long long* ext_off,
                                    unsigned e0, unsigned e1, long long ext_base, const T* src, T* dst) {
  const int lane = threadIdx.x & 31;
  unsigned e = e0 + (unsigned)((blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x) >> 5);
  const unsigned stride = (unsigned)((gridDim.x * (unsigned long long)blockDim.x) >> 5);
  for (; e < e1; e += stride) {
    unsigned r = ext_to_int[e];
    int s = key_slot(t.row_key[r]);
    SlotInfo si = t.sinfo[s];
    long long ie = row_elem(si, r);
    long long xe = ext_elem(ext_off, t.uniform_dim, e) - ext_base;
    for (int j = lane; j < si.dim; j += 32) {
      if (kToInt)
        dst[ie + j] = src[xe + j];
      else
        dst[xe + j] = src[ie + j];
    }
  }
}

// The f16 copy of a master-copy table: every element rounded to nearest-even.
__global__ void half_copy_kernel(const float* __restrict__ w, __half* __restrict__ h, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    h[i] = __float2half_rn(w[i]);
}

__global__ void fill_f32_kernel(float* p, long long n, float v) {
  long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  for (; i < n; i += (long long)gridDim.x * blockDim.x) p[i] = v;
}

__global__ void export_keys_kernel(const long long* row_key, const unsigned* ext_to_int, unsigned e0, unsigned e1,
                                   long long* out) {
  unsigned e = e0 + blockIdx.x * blockDim.x + threadIdx.x;
  for (; e < e1; e += gridDim.x * blockDim.x) out[e - e0] = row_key[ext_to_int[e]];
}

__global__ void slots_kernel(const Slot* slots, long long p0, long long p1, long long* skey, long long* srow) {
  long long p = p0 + blockIdx.x * (long long)blockDim.x + threadIdx.x;
  for (; p < p1; p += (long long)gridDim.x * blockDim.x) {
    Slot s = slots[p];
    if (skey) skey[p - p0] = s.key;
    if (srow) srow[p - p0] = s.key == kEmptyKey ? -1 : (long long)s.ext;
  }
}

// Selected keys-array rows to a dense [n, max_dim] buffer (zero padded).
template <typename T>
__global__ void export_rows_kernel(TableView t, const unsigned* ext_to_int, const long long* __restrict__ rows,
                                   long long n, unsigned n_keys, T* __restrict__ vout, float* __restrict__ aout,
                                   int acc_per_row) {
  const int lane = threadIdx.x & 31;
  const T* W = static_cast<const T*>(t.W);
  long long i = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long stride = ((long long)gridDim.x * blockDim.x) >> 5;
  for (; i < n; i += stride) {
    const long long e = rows[i];
    const bool ok = e >= 0 && e < (long long)n_keys;
    if (!ok && lane == 0) atomicOr(t.flags, EMB_FLAG_BAD_ROW);
    int D = 0;
    long long ie = 0;
    unsigned r = 0;
    if (ok) {
      r = ext_to_int[e];
      const SlotInfo si = t.sinfo[key_slot(t.row_key[r])];
      D = si.dim;
      ie = row_elem(si, r);
    }
    for (int j = lane; j < t.max_dim; j += 32) {
      const bool in = j < D;
      if (vout) vout[i * t.max_dim + j] = in ? W[ie + j] : T(0);
      if (aout && !acc_per_row) aout[i * t.max_dim + j] = in ? t.ACC[ie + j] : 0.f;
    }
    if (aout && acc_per_row && lane == 0) aout[i] = ok ? t.ACC[r] : 0.f;
  }
}

// Kernel P: the probe alone, one thread per key.
__global__ void resolve_kernel(TableView t, const long long* __restrict__ keys, long long n, long long* slot_out,
                               long long* row_out) {
  long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  for (; i < n; i += (long long)gridDim.x * blockDim.x) {
    unsigned row = 0, ext = 0;
    unsigned long long h = 0;
    bool hit = probe(t, keys[i], &row, &ext, &h);
    if (slot_out) slot_out[i] = hit ? (long long)h : -1;
    if (row_out) row_out[i] = hit ? (long long)ext : -1;
  }
}

static int grid_for(long long work, int per_block) {
  long long g = (work + per_block - 1) / per_block;
  long long cap = (long long)sm_count() * 16;
  if (g > cap) g = cap;
  return (int)std::max(1LL, g);
}

static bool is_device_ptr(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

static long long ext_elem_h(const emb_table* t, const std::vector<long long>& off, unsigned e) {
  return off.empty() ? (long long)e * t->uniform_dim : off[e];
}

// One f32 per key between keys-array order (src or dst) and internal row order.
template <bool kToTable>
__global__ void permute_keys_kernel(const unsigned* __restrict__ ext_to_int, unsigned n, const float* __restrict__ src,
                                    float* __restrict__ dst) {
  for (unsigned e = blockIdx.x * blockDim.x + threadIdx.x; e < n; e += gridDim.x * blockDim.x) {
    if (kToTable) dst[ext_to_int[e]] = src[e];
    else dst[e] = src[ext_to_int[e]];
  }
}

// Move one f32 per key (row-wise accumulators) between a caller buffer in
// keys-array order (host or device) and the table's array in internal order.
static emb_status move_keyvals(const emb_table* t, const float* user, float* table_arr, bool to_table,
                               cudaStream_t st) {
  const unsigned n = (unsigned)t->st.n_keys;
  if (n == 0) return EMB_OK;
  const bool dev = is_device_ptr(user);
  float* buf = (float*)user;
  if (!dev) {
    EMB_CUDA(dmalloc((void**)&buf, (size_t)n * 4));
    if (to_table) {
      cudaError_t ce = cudaMemcpyAsync(buf, user, (size_t)n * 4, cudaMemcpyHostToDevice, st);
      if (ce != cudaSuccess) {
        dfree(buf);
        return cuda_fail(ce, "cudaMemcpyAsync(accumulators to device)");
      }
    }
  }
  if (to_table)
    permute_keys_kernel<true><<<grid_for(n, 256), 256, 0, st>>>(t->ext_to_int_d, n, buf, table_arr);
  else
    permute_keys_kernel<false><<<grid_for(n, 256), 256, 0, st>>>(t->ext_to_int_d, n, table_arr, buf);
  cudaError_t ce = cudaGetLastError();
  if (ce == cudaSuccess && !dev && !to_table)
    ce = cudaMemcpyAsync((void*)user, buf, (size_t)n * 4, cudaMemcpyDeviceToHost, st);
  if (ce == cudaSuccess && !dev) ce = cudaStreamSynchronize(st);
  if (!dev) dfree(buf);
  if (ce != cudaSuccess) return cuda_fail(ce, "moving per-key accumulators");
  return EMB_OK;
}

// Move ragged rows between a caller buffer in keys-array order (host or
// device) and a table array in internal order, in chunks through a staging
// buffer when the caller's buffer is host memory.
static emb_status move_rows(const emb_table* t, const void* user,
                            void* table_arr, size_t esz, bool to_table, cudaStream_t st) {
  const unsigned n = (unsigned)t->st.n_keys;
  if (n == 0) return EMB_OK;
  const bool dev = is_device_ptr(user);
  const long long kStageElems = 32LL << 20;
  void* stage = nullptr;
  if (!dev) EMB_CUDA(dmalloc(&stage, (size_t)std::min<long long>(kStageElems, t->st.n_elems) * esz));
  emb_status rc = EMB_OK;
  TableView v = t->view();
  const std::vector<long long>& ext_off_h = t->ext_elem_off_h;
  unsigned e0 = 0;
  while (e0 < n) {
    unsigned e1 = e0;
    long long base = ext_elem_h(t, ext_off_h, e0);
    if (dev) {
      e1 = n;
    } else {
      // rows fitting in the staging buffer (a row is at most EMB_MAX_DIM elements)
      unsigned lo = e0 + 1, hi = n;
      while (lo < hi) {
        unsigned mid = lo + (hi - lo + 1) / 2;
        if (ext_elem_h(t, ext_off_h, mid) - base <= kStageElems) lo = mid; else hi = mid - 1;
      }
      e1 = lo;
    }
    long long end = ext_elem_h(t, ext_off_h, e1);
    size_t bytes = (size_t)(end - base) * esz;
    const char* ubase = (const char*)user + (size_t)base * esz;
    void* buf = dev ? (void*)ubase : stage;
    cudaError_t ce = cudaSuccess;
    if (!dev && to_table) ce = cudaMemcpyAsync(stage, ubase, bytes, cudaMemcpyHostToDevice, st);
    if (ce != cudaSuccess) { rc = cuda_fail(ce, "cudaMemcpyAsync(rows to device)"); break; }
    int grid = grid_for((long long)(e1 - e0) * 32, 256);
    if (esz == 2) {
      if (to_table)
        permute_rows_kernel<unsigned short, true><<<grid, 256, 0, st>>>(v, t->ext_to_int_d, t->ext_elem_off_d, e0, e1,
                                                                        base, (const unsigned short*)buf, (unsigned short*)table_arr);
      else
        permute_rows_kernel<unsigned short, false><<<grid, 256, 0, st>>>(v, t->ext_to_int_d, t->ext_elem_off_d, e0, e1,
                                                                         base, (const unsigned short*)table_arr, (unsigned short*)buf);
    } else {
      if (to_table)
        permute_rows_kernel<unsigned, true><<<grid, 256, 0, st>>>(v, t->ext_to_int_d, t->ext_elem_off_d, e0, e1, base,
                                                                  (const unsigned*)buf, (unsigned*)table_arr);
      else
        permute_rows_kernel<unsigned, false><<<grid, 256, 0, st>>>(v, t->ext_to_int_d, t->ext_elem_off_d, e0, e1, base,
                                                                   (const unsigned*)table_arr, (unsigned*)buf);
    }
    ce = cudaGetLastError();
    if (ce != cudaSuccess) { rc = cuda_fail(ce, "permute_rows_kernel launch"); break; }
    if (!dev && !to_table) {
      ce = cudaMemcpyAsync((void*)ubase, stage, bytes, cudaMemcpyDeviceToHost, st);
      if (ce != cudaSuccess) { rc = cuda_fail(ce, "cudaMemcpyAsync(rows to host)"); break; }
    }
    if (!dev) {
      ce = cudaStreamSynchronize(st);  // the staging buffer is reused
      if (ce != cudaSuccess) { rc = cuda_fail(ce, "cudaStreamSynchronize"); break; }
    }
    e0 = e1;
  }
  if (stage) {
    cudaStreamSynchronize(st);
    dfree(stage);
  }
  return rc;
}

void free_table(emb_table* t) {
  if (!t) return;
  dfree(t->slots_d);
  dfree(t->sinfo_d);
  dfree(t->W_d);
  dfree(t->W16_d);
  dfree(t->ACC_d);
  dfree(t->Z_d);
  dfree(t->row_key_d);
  dfree(t->int_to_ext_d);
  dfree(t->ext_to_int_d);
  dfree(t->ext_elem_off_d);
  dfree(t->flags_d);
  delete t;
}

template <typename T>
emb_status dalloc_copy(T** dst, const T* src, size_t count, cudaStream_t st, uint64_t* bytes) {
  size_t b = std::max<size_t>(count, 1) * sizeof(T);
  EMB_CUDA(dmalloc((void**)dst, b));
  *bytes += b;
  if (src && count) EMB_CUDA(cudaMemcpyAsync(*dst, src, count * sizeof(T), cudaMemcpyHostToDevice, st));
  return EMB_OK;
}

// The part of table creation after the slot layout and the row maps are on
// the device: the flag word, weights (from values, in keys-array order, or
// zeros), the f16 copy of master-copy tables, accumulators (acc or
// desc->acc_init) and FTRL's z; synchronises the stream.
emb_status finish_table(emb_table* t, const emb_table_desc* desc, const void* values, const float* acc,
                        cudaStream_t st, uint64_t* bytes_io) {
  uint64_t& bytes = *bytes_io;
  emb_status r;
  const size_t esz = t->st.wdtype == EMB_F16 ? 2 : 4;
  if ((r = dalloc_copy(&t->flags_d, (const unsigned*)nullptr, 1, st, &bytes)) != EMB_OK) return r;
  EMB_CUDA(cudaMemsetAsync(t->flags_d, 0, sizeof(unsigned), st));
  const size_t ne = (size_t)std::max<long long>(t->st.n_elems, 1);
  EMB_CUDA(dmalloc(&t->W_d, ne * esz));
  bytes += ne * esz;
  const bool rowwise = desc->optimizer == EMB_OPT_ROWWISE_ADAGRAD;
  const size_t na = rowwise ? (size_t)std::max<long long>(t->st.n_keys, 1) : ne;  // accumulators
  EMB_CUDA(dmalloc((void**)&t->ACC_d, na * 4));
  bytes += na * 4;
  t->st.device_bytes = bytes;
  if (values) {
    if ((r = move_rows(t, values, t->W_d, esz, true, st)) != EMB_OK) return r;
  } else {
    EMB_CUDA(cudaMemsetAsync(t->W_d, 0, ne * esz, st));
  }
  if (t->st.wdtype == EMB_F16_MASTER) {  // W holds the f32 master; the forward reads its f16 copy
    EMB_CUDA(dmalloc(&t->W16_d, ne * 2));
    bytes += ne * 2;
    t->st.device_bytes = bytes;
    half_copy_kernel<<<grid_for((long long)ne, 256), 256, 0, st>>>((const float*)t->W_d, (__half*)t->W16_d,
                                                                   (long long)ne);
    EMB_CUDA(cudaGetLastError());
  }
  if (acc) {
    if ((r = rowwise ? move_keyvals(t, acc, t->ACC_d, true, st) : move_rows(t, acc, t->ACC_d, 4, true, st)) != EMB_OK)
      return r;
  } else {
    fill_f32_kernel<<<grid_for((long long)na, 256), 256, 0, st>>>(t->ACC_d, (long long)na, desc->acc_init);
    EMB_CUDA(cudaGetLastError());
  }
  if (desc->optimizer == EMB_OPT_FTRL) {  // FTRL's z starts at zero (emb_table_import_z sets it)
    EMB_CUDA(dmalloc((void**)&t->Z_d, ne * 4));
    bytes += ne * 4;
    t->st.device_bytes = bytes;
    EMB_CUDA(cudaMemsetAsync(t->Z_d, 0, ne * 4, st));
  }
  EMB_CUDA(cudaStreamSynchronize(st));
  return EMB_OK;
}

}  // namespace emb

using namespace emb;

extern "C" {

const char* emb_status_string(emb_status s) {
  switch (s) {
    case EMB_OK: return "ok";
    case EMB_ERR_INVALID_ARG: return "invalid argument";
    case EMB_ERR_CUDA: return "CUDA error";
    case EMB_ERR_OOM: return "out of memory";
    case EMB_ERR_DUP_KEY: return "duplicate key";
    case EMB_ERR_RESERVED_KEY: return "reserved key";
    case EMB_ERR_LOAD_FACTOR: return "capacity/load factor";
    case EMB_ERR_WORKSPACE: return "workspace too small";
    case EMB_ERR_DEVICE_FLAG: return "device flag raised";
    case EMB_ERR_UNSUPPORTED: return "unsupported size";
  }
  return "unknown status";
}

const char* emb_last_error(void) { return g_last_error.c_str(); }

emb_status emb_table_plan(const emb_table_desc* desc, const int64_t* keys_h, int64_t n_keys, emb_table_stats* out,
                          int64_t* slot_key_h, int64_t* slot_row_h) {
  HostPlan P;
  const bool want = slot_key_h || slot_row_h;
  emb_status rc = build_plan(desc, keys_h, n_keys, P, want);
  if (rc != EMB_OK) return rc;
  if (out) *out = P.st;
  if (want) {
    for (size_t p = 0; p < P.slots.size(); ++p) {
      const Slot& s = P.slots[p];
      if (slot_key_h) slot_key_h[p] = s.key;
      if (slot_row_h) slot_row_h[p] = s.key == kEmptyKey ? -1 : (int64_t)s.ext;
    }
  }
  return EMB_OK;
}

emb_status emb_table_create(const emb_table_desc* desc, const int64_t* keys_h, int64_t n_keys, const void* values,
                            const float* acc, void* stream, emb_table** out) {
  if (!out) return fail(EMB_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  HostPlan P;
  emb_status rc = build_plan(desc, keys_h, n_keys, P, true);
  if (rc != EMB_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  emb_table* t = new (std::nothrow) emb_table();
  if (!t) return fail(EMB_ERR_OOM, "host allocation failed");
  cudaGetDevice(&t->device);
  t->optimizer = (int)desc->optimizer;
  t->st = P.st;
  t->sinfo_h = P.sinfo;
  t->uniform_dim = P.ext_elem_off.empty() ? P.dims[0] : 0;
  t->ext_elem_off_h.swap(P.ext_elem_off);
  uint64_t bytes = 0;
  auto body = [&]() -> emb_status {
    emb_status r;
    // the prepared table is flashed to global memory in one block
    if ((r = dalloc_copy(&t->slots_d, P.slots.data(), P.slots.size(), st, &bytes)) != EMB_OK) return r;
    if ((r = dalloc_copy(&t->sinfo_d, P.sinfo.data(), P.sinfo.size(), st, &bytes)) != EMB_OK) return r;
    if ((r = dalloc_copy(&t->row_key_d, P.row_key.data(), P.row_key.size(), st, &bytes)) != EMB_OK) return r;
    if ((r = dalloc_copy(&t->int_to_ext_d, P.int_to_ext.data(), P.int_to_ext.size(), st, &bytes)) != EMB_OK) return r;
    if ((r = dalloc_copy(&t->ext_to_int_d, P.ext_to_int.data(), P.ext_to_int.size(), st, &bytes)) != EMB_OK) return r;
    if (!t->ext_elem_off_h.empty() &&
        (r = dalloc_copy(&t->ext_elem_off_d, (const long long*)t->ext_elem_off_h.data(), t->ext_elem_off_h.size(), st,
                         &bytes)) != EMB_OK)
      return r;
    return finish_table(t, desc, values, acc, st, &bytes);
  };
  rc = body();
  if (rc != EMB_OK) {
    cudaStreamSynchronize(st);
    free_table(t);
    return rc;
  }
  *out = t;
  return EMB_OK;
}

emb_status emb_table_destroy(emb_table* table) {
  if (!table) return fail(EMB_ERR_INVALID_ARG, "table is NULL");
  free_table(table);
  return EMB_OK;
}

emb_status emb_table_get_stats(const emb_table* table, emb_table_stats* out) {
  if (!table || !out) return fail(EMB_ERR_INVALID_ARG, "NULL argument");
  *out = table->st;
  return EMB_OK;
}

emb_status emb_resolve(const emb_table* table, const int64_t* keys_d, int64_t n, int64_t* slot_out_d,
                       int64_t* row_out_d, void* stream) {
  if (!table || n < 0 || (n > 0 && !keys_d)) return fail(EMB_ERR_INVALID_ARG, "bad resolve arguments");
  if (n == 0) return EMB_OK;
  resolve_kernel<<<grid_for(n, 256), 256, 0, (cudaStream_t)stream>>>(
      table->view(), (const long long*)keys_d, n, (long long*)slot_out_d, (long long*)row_out_d);
  EMB_CUDA(cudaGetLastError());
  return EMB_OK;
}

emb_status emb_table_export(const emb_table* table, int64_t* keys_out, void* values_out, float* acc_out,
                            void* stream) {
  if (!table) return fail(EMB_ERR_INVALID_ARG, "table is NULL");
  cudaStream_t st = (cudaStream_t)stream;
  const unsigned n = (unsigned)table->st.n_keys;
  const size_t esz = table->st.wdtype == EMB_F16 ? 2 : 4;
  emb_status r;
  if (values_out && (r = move_rows(table, values_out, table->W_d, esz, false, st)) != EMB_OK) return r;
  if (acc_out) {
    r = table->optimizer == EMB_OPT_ROWWISE_ADAGRAD ? move_keyvals(table, acc_out, table->ACC_d, false, st)
                                                    : move_rows(table, acc_out, table->ACC_d, 4, false, st);
    if (r != EMB_OK) return r;
  }
  if (keys_out && n) {
    if (is_device_ptr(keys_out)) {
      export_keys_kernel<<<grid_for(n, 256), 256, 0, st>>>(table->row_key_d, table->ext_to_int_d, 0, n,
                                                           (long long*)keys_out);
      EMB_CUDA(cudaGetLastError());
    } else {
      long long* tmp = nullptr;
      EMB_CUDA(dmalloc((void**)&tmp, (size_t)n * 8));
      export_keys_kernel<<<grid_for(n, 256), 256, 0, st>>>(table->row_key_d, table->ext_to_int_d, 0, n, tmp);
      cudaError_t e = cudaGetLastError();
      if (e == cudaSuccess) e = cudaMemcpyAsync(keys_out, tmp, (size_t)n * 8, cudaMemcpyDeviceToHost, st);
      if (e == cudaSuccess) e = cudaStreamSynchronize(st);
      dfree(tmp);
      if (e != cudaSuccess) return cuda_fail(e, "export keys");
    }
  }
  EMB_CUDA(cudaStreamSynchronize(st));
  return EMB_OK;
}

emb_status emb_table_export_z(const emb_table* table, float* z_out, void* stream) {
  if (!table || !z_out) return fail(EMB_ERR_INVALID_ARG, "NULL argument");
  if (!table->Z_d) return fail(EMB_ERR_INVALID_ARG, "not an FTRL table");
  cudaStream_t st = (cudaStream_t)stream;
  emb_status r = move_rows(table, z_out, table->Z_d, 4, false, st);
  if (r != EMB_OK) return r;
  EMB_CUDA(cudaStreamSynchronize(st));
  return EMB_OK;
}

emb_status emb_table_import_z(emb_table* table, const float* z_in, void* stream) {
  if (!table || !z_in) return fail(EMB_ERR_INVALID_ARG, "NULL argument");
  if (!table->Z_d) return fail(EMB_ERR_INVALID_ARG, "not an FTRL table");
  cudaStream_t st = (cudaStream_t)stream;
  emb_status r = move_rows(table, z_in, table->Z_d, 4, true, st);
  if (r != EMB_OK) return r;
  EMB_CUDA(cudaStreamSynchronize(st));
  return EMB_OK;
}

emb_status emb_table_export_rows(const emb_table* table, const int64_t* ext_rows_d, int64_t n, void* values_out_d,
                                 float* acc_out_d, void* stream) {
  if (!table || n < 0 || (n > 0 && !ext_rows_d)) return fail(EMB_ERR_INVALID_ARG, "bad export_rows arguments");
  if (n == 0 || (!values_out_d && !acc_out_d)) return EMB_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const int grid = grid_for(n * 32, 256);
  const unsigned nk = (unsigned)table->st.n_keys;
  const int rw = table->optimizer == EMB_OPT_ROWWISE_ADAGRAD ? 1 : 0;
  if (table->st.wdtype == EMB_F16)
    export_rows_kernel<unsigned short><<<grid, 256, 0, st>>>(table->view(), table->ext_to_int_d,
                                                             (const long long*)ext_rows_d, n, nk,
                                                             (unsigned short*)values_out_d, acc_out_d, rw);
  else
    export_rows_kernel<unsigned><<<grid, 256, 0, st>>>(table->view(), table->ext_to_int_d,
                                                       (const long long*)ext_rows_d, n, nk, (unsigned*)values_out_d,
                                                       acc_out_d, rw);
  EMB_CUDA(cudaGetLastError());
  return EMB_OK;
}

emb_status emb_table_slots(const emb_table* table, int64_t* slot_key_out, int64_t* slot_row_out, void* stream) {
  if (!table) return fail(EMB_ERR_INVALID_ARG, "table is NULL");
  cudaStream_t st = (cudaStream_t)stream;
  const long long cap = table->st.capacity;
  const bool dk = !slot_key_out || is_device_ptr(slot_key_out);
  const bool dr = !slot_row_out || is_device_ptr(slot_row_out);
  if (dk && dr) {
    slots_kernel<<<grid_for(cap, 256), 256, 0, st>>>(table->slots_d, 0, cap, (long long*)slot_key_out,
                                                     (long long*)slot_row_out);
    EMB_CUDA(cudaGetLastError());
    EMB_CUDA(cudaStreamSynchronize(st));
    return EMB_OK;
  }
  const long long chunk = 16LL << 20;
  long long* tmp = nullptr;
  EMB_CUDA(dmalloc((void**)&tmp, (size_t)std::min(chunk, cap) * 16));
  cudaError_t e = cudaSuccess;
  for (long long p0 = 0; p0 < cap && e == cudaSuccess; p0 += chunk) {
    long long p1 = std::min(cap, p0 + chunk), m = p1 - p0;
    slots_kernel<<<grid_for(m, 256), 256, 0, st>>>(table->slots_d, p0, p1, tmp, tmp + m);
    e = cudaGetLastError();
    if (e == cudaSuccess && slot_key_out)
      e = cudaMemcpyAsync(slot_key_out + p0, tmp, (size_t)m * 8, cudaMemcpyDefault, st);
    if (e == cudaSuccess && slot_row_out)
      e = cudaMemcpyAsync(slot_row_out + p0, tmp + m, (size_t)m * 8, cudaMemcpyDefault, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  }
  dfree(tmp);
  if (e != cudaSuccess) return cuda_fail(e, "emb_table_slots");
  return EMB_OK;
}

emb_status emb_debug_fail_device_alloc(int64_t after) {
  g_fail_after.store(after < 0 ? -1 : (long long)after);
  return EMB_OK;
}

int64_t emb_debug_live_device_allocs(void) { return (int64_t)g_live_allocs.load(); }

emb_status emb_debug_set_probe_bound(emb_table* table, int64_t bound) {
  if (!table || bound < 1 || bound > table->st.max_cluster + 1)
    return fail(EMB_ERR_INVALID_ARG, "probe bound must be in [1, max_cluster + 1]");
  table->st.probe_bound = bound;
  return EMB_OK;
}

emb_status emb_check_device_flag(emb_table* table, void* stream, uint32_t* flags_out) {
  if (!table) return fail(EMB_ERR_INVALID_ARG, "table is NULL");
  cudaStream_t st = (cudaStream_t)stream;
  unsigned f = 0;
  EMB_CUDA(cudaStreamSynchronize(st));
  EMB_CUDA(cudaMemcpy(&f, table->flags_d, sizeof f, cudaMemcpyDeviceToHost));
  EMB_CUDA(cudaMemset(table->flags_d, 0, sizeof f));
  if (flags_out) *flags_out = f;
  if (f) {
    char buf[96];
    std::snprintf(buf, sizeof buf, "device flag bits 0x%x (probe bound 1, offsets 2, slot mismatch 4)", f);
    return fail(EMB_ERR_DEVICE_FLAG, buf);
  }
  return EMB_OK;
}

}  // extern "C"
