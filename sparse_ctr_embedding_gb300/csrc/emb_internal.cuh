// Internal definitions shared by the library's translation units.
//
// Device data layout of one table (all owned by emb_table):
//   slots   Slot[capacity]   16-byte entries {int64 key; u32 row; u32 ext},
//                            key == -1 marks an empty slot.  row is the
//                            internal (slot-major) row, ext the key's index in
//                            the keys array given at creation.
//   W       wdtype[n_elems]  weights, internal row order.  Rows of one feature
//                            slot are contiguous (slot-major), so a row's
//                            first element is elem_base[s] + (row - row_base[s]) * dim[s].
//   ACC     f32[n_elems]     Adagrad accumulators, same layout as W;
//                            f32[n_rows] (one per internal row) for
//                            EMB_OPT_ROWWISE_ADAGRAD tables.
//   W16     f16[n_elems]     EMB_F16_MASTER tables only: the f16 copy of W
//                            (then the f32 master) that the forward reads.
//   Z       f32[n_elems]     EMB_OPT_FTRL tables only: FTRL's z (ACC is n).
//   row_key int64[n_rows]    key of each internal row.
//   int_to_ext / ext_to_int  u32[n_rows] row-order permutations.
//   flags   u32              EMB_FLAG_* bits raised by kernels.
// Slot-major rows keep every gradient row of one feature slot (one column
// block of grad_out) together after the backward's sort by row, so the
// segmented reduction reads a working set of one slot's grad_out columns.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <vector>

#include "../../include/emb_gb300.h"

namespace emb {

constexpr long long kEmptyKey = -1LL;

struct __align__(16) Slot {
  long long key;
  unsigned int row;
  unsigned int ext;
};
static_assert(sizeof(Slot) == 16, "slot entry is 16 bytes");

struct SlotInfo {
  int dim;
  int col;                 // first column of this slot in the pooled output
  unsigned int row_base;   // first internal row
  unsigned int n_rows;
  long long elem_base;     // first weight element
};

// Everything a kernel needs to know about the table, passed by value.
struct TableView {
  const Slot* slots;
  unsigned long long mask;  // capacity - 1
  int probe_bound;          // max_cluster + 1
  int n_slots;
  int sum_dims;
  int uniform_dim;          // dim shared by all slots, or 0 if dims differ
  int max_dim;
  unsigned int n_rows;
  const SlotInfo* sinfo;    // [n_slots]
  void* W;
  float* ACC;
  float* Z;                 // FTRL tables: the second state array; else NULL
  __half* W16;              // master-copy tables: the f16 copy of W; else NULL
  const long long* row_key;
  unsigned int* flags;
};

// ------------------------------------------------------------------ device helpers

// MurmurHash3 64-bit finalizer (Appleby, public domain): the table's hash.
__device__ __forceinline__ unsigned long long fmix64(unsigned long long k) {
  k ^= k >> 33;
  k *= 0xff51afd7ed558ccdULL;
  k ^= k >> 33;
  k *= 0xc4ceb9fe1a85ec53ULL;
  k ^= k >> 33;
  return k;
}

// One 16-byte read-only load of a slot entry (the table never changes during
// a step): key, then row (low 32 bits) and ext (high 32 bits).
__device__ __forceinline__ void ld_slot(const Slot* p, long long& key, unsigned long long& row_ext) {
  asm("ld.global.nc.v2.u64 {%0, %1}, [%2];" : "=l"(key), "=l"(row_ext) : "l"(p));
}

// Bounded linear probe.  Returns true and the entry on a hit.  A key equal to
// the empty sentinel never hits.  More than probe_bound inspected slots can
// only happen on a corrupted table: the flag is raised and the key misses.
__device__ __forceinline__ bool probe(const TableView& t, long long key, unsigned int* row,
                                      unsigned int* ext, unsigned long long* slot_idx) {
  if (key == kEmptyKey) return false;
  unsigned long long h = fmix64((unsigned long long)key) & t.mask;
  for (int p = 0; p < t.probe_bound; ++p) {
    long long k;
    unsigned long long re;
    ld_slot(t.slots + h, k, re);
    if (k == kEmptyKey) return false;
    if (k == key) {
      *row = (unsigned int)re;
      *ext = (unsigned int)(re >> 32);
      *slot_idx = h;
      return true;
    }
    h = (h + 1) & t.mask;
  }
  atomicOr(t.flags, EMB_FLAG_PROBE_BOUND);
  return false;
}

__device__ __forceinline__ int key_slot(long long key) { return (int)(((unsigned long long)key) >> 48); }

// First weight element of an internal row of slot s.
__device__ __forceinline__ long long row_elem(const SlotInfo& si, unsigned int row) {
  return si.elem_base + (long long)(row - si.row_base) * si.dim;
}

// ------------------------------------------------------------------ host side

struct HostPlan {
  int n_slots = 0;
  std::vector<int32_t> dims;
  emb_dtype wdtype = EMB_F32;
  int64_t n_keys = 0, cap = 0;
  std::vector<Slot> slots;                 // [cap]
  std::vector<SlotInfo> sinfo;             // [n_slots]
  std::vector<uint32_t> ext_to_int;        // [n]
  std::vector<uint32_t> int_to_ext;        // [n]
  std::vector<long long> row_key;          // [n]
  std::vector<long long> ext_elem_off;     // [n+1]
  emb_table_stats st{};
};

}  // namespace emb

struct emb_table {
  int device = 0;
  emb_table_stats st{};
  std::vector<emb::SlotInfo> sinfo_h;
  emb::Slot* slots_d = nullptr;
  emb::SlotInfo* sinfo_d = nullptr;
  void* W_d = nullptr;      // weights (the f32 master for EMB_F16_MASTER tables)
  void* W16_d = nullptr;    // EMB_F16_MASTER tables: the f16 copy the forward reads
  float* ACC_d = nullptr;
  float* Z_d = nullptr;     // FTRL tables: z
  int optimizer = EMB_OPT_ADAGRAD;
  long long* row_key_d = nullptr;
  unsigned int* int_to_ext_d = nullptr;
  unsigned int* ext_to_int_d = nullptr;
  long long* ext_elem_off_d = nullptr;  // ragged tables only
  unsigned int* flags_d = nullptr;
  int uniform_dim = 0;
  std::vector<long long> ext_elem_off_h;  // ragged tables only: host copy for chunked transfers
  void* phase_events[EMB_BWD_PHASES] = {};  // caller-owned cudaEvent_t, see emb_bwd_phase_events
  int n_phase_events = 0;
  // the last emb_lookup_fwd_record: which workspace holds its (row, bag) pairs
  const void* rec_ws = nullptr;
  long long rec_nnz = -1, rec_bags = -1;
  int rec_pool = -1;
  bool rec_sorted = false;  // the recording forward also sorted the pairs (emb_lookup_fwd_dedup)

  emb::TableView view() const {
    emb::TableView v;
    v.slots = slots_d;
    v.mask = (unsigned long long)st.capacity - 1ULL;
    v.probe_bound = (int)st.probe_bound;
    v.n_slots = st.n_slots;
    v.sum_dims = st.sum_dims;
    v.uniform_dim = uniform_dim;
    v.max_dim = st.max_dim;
    v.n_rows = (unsigned int)st.n_keys;
    v.sinfo = sinfo_d;
    v.W = W_d;
    v.ACC = ACC_d;
    v.Z = Z_d;
    v.W16 = (__half*)W16_d;
    v.row_key = row_key_d;
    v.flags = flags_d;
    return v;
  }
  // The view the forward gathers from: the f16 copy of a master-copy table.
  emb::TableView fwd_view() const {
    emb::TableView v = view();
    if (W16_d) v.W = W16_d;
    return v;
  }
  // Element type the forward reads.
  bool fwd_half() const { return st.wdtype == EMB_F16 || st.wdtype == EMB_F16_MASTER; }
};

namespace emb {
// error reporting and launch helpers (emb_table.cu)
emb_status fail(emb_status s, const std::string& msg);
emb_status cuda_fail(cudaError_t e, const char* what);
int sm_count();
// every device allocation of the library (counted; see emb_debug_fail_device_alloc)
cudaError_t dmalloc(void** p, size_t bytes);
void dfree(void* p);
// table creation steps shared by the host and the device build (emb_table.cu)
emb_status check_desc(const emb_table_desc* d, int64_t n, int64_t* cap_out, int* max_dim_out,
                      long long* sum_dims_out);
emb_status finish_table(emb_table* t, const emb_table_desc* desc, const void* values, const float* acc,
                        cudaStream_t st, uint64_t* bytes_io);
void free_table(emb_table* t);
// sort and scan building blocks (emb_bwd.cu)
size_t pair_sort_scratch_bytes(unsigned n);
cudaError_t pair_sort(unsigned* kA, unsigned* vA, unsigned* kB, unsigned* vB, unsigned n, int bits, void* scratch,
                      cudaStream_t st, bool* in_b);
cudaError_t launch_scan_u32(const unsigned* in, unsigned* out, size_t n, unsigned* partials, cudaStream_t st);
}  // namespace emb

#define EMB_CUDA(call)                                        \
  do {                                                        \
    cudaError_t e_ = (call);                                  \
    if (e_ != cudaSuccess) return emb::cuda_fail(e_, #call);  \
  } while (0)
