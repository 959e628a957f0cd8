// CPU oracle for the unified-hash-table embedding step.
//
// TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
// and the benchmark's CPU-baseline leg load this library.  It is a plain,
// slow, single-threaded restatement of what the step computes, written
// independently of the CUDA path (it includes none of its headers and shares
// no helper with it), in double precision wherever the method leaves the
// precision open.  Built with -ffp-contract=off so that every float expression
// rounds exactly as written on every host architecture.
//
// Sources (page title, then the passage):
//  [TPCG]  Tencent PCG DataFun talk on GPU recommendation-training frameworks,
//          "各阶段优化详细介绍" (the insert-free GPU hashtable: the table is
//          prepared beforehand from a group's deduplicated keys and flashed to
//          global memory whole, no insert) and "计算优化" (Unified Hash Table:
//          int64 key, low 48 bits the real key, high 16 bits the table id; one
//          lookup kernel and one backward kernel for all features).
//  [JD]    JD ads large-scale sparse training article, section 3.2.1 (sparse
//          optimizers: Adagrad keeps a per-parameter accumulated sum of squared
//          gradients as an adaptive learning rate; the update is element-wise;
//          features absent from the batch leave parameters and state
//          untouched) and section 4.2.1 (EmbeddingBag sum/mean pooling of the
//          looked-up vectors per sample).
//  [META]  MetaApp DeepRec article, section 3.3 (Adagrad, learning rate 0.01).
//  The hash (MurmurHash3 fmix64), the probe scheme (linear probing over a
//  power-of-two table) and the Adagrad closed form
//      acc += g*g;  w -= lr * g / (sqrt(acc) + eps)
//  are fixed by the step's specification, not by the pages.
//
// Readings where the pages are silent (each also listed in the design notes):
//  * slots are assigned by inserting keys one by one in keys-array order;
//  * the empty-slot sentinel is the all-ones int64 (-1), which is never a key;
//  * a bag (sample b, slot s) pools only table keys whose slot field is s;
//    other keys contribute nothing (misses pool as zero vectors);
//  * mean pooling divides by the bag length L counting misses; L = 0 gives 0;
//  * a key repeated inside one bag counts once per occurrence, in the pooled
//    sum and in the gradient.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <unordered_map>
#include <unordered_set>
#include <vector>

namespace {

constexpr int64_t kEmpty = -1;  // all ones

enum : int {
  ORC_OK = 0,
  ORC_INVALID = 1,
  ORC_DUP_KEY = 2,
  ORC_RESERVED_KEY = 3,
  ORC_BAD_SLOT = 4,
  ORC_DISAGREE = 5,
  ORC_MISSING_ROW = 6,
};

// MurmurHash3 64-bit finalizer (Austin Appleby, MurmurHash3, public domain).
uint64_t fmix64(uint64_t k) {
  k ^= k >> 33;
  k *= 0xff51afd7ed558ccdULL;
  k ^= k >> 33;
  k *= 0xc4ceb9fe1a85ec53ULL;
  k ^= k >> 33;
  return k;
}

int slot_of_key(int64_t key) { return (int)(((uint64_t)key) >> 48); }  // [TPCG] 计算优化

}  // namespace

struct orc_table {
  int64_t n = 0, cap = 0;
  int n_slots = 0;
  std::vector<int32_t> dims;
  std::vector<int64_t> keys;                    // keys-array order
  std::unordered_map<int64_t, int64_t> row_of;  // key -> keys-array index
  std::vector<int64_t> slot_key, slot_row;      // simulated insert-free layout
  std::vector<int64_t> elem_off;                // per row, ragged values array
  int64_t max_probe = 0;    // longest probe sequence of an inserted key
  int64_t sum_probe = 0;    // sum of probe lengths of inserted keys
  int64_t max_cluster = 0;  // longest run of occupied slots
};

struct orc_grad {
  std::vector<int64_t> keys, rows, goff;
  std::vector<double> G, A;
};

extern "C" {

uint64_t orc_fmix64(uint64_t k) { return fmix64(k); }

// Build the prepared table of [TPCG] 各阶段优化: all keys known up front, one
// sequential insertion each, in keys-array order, then never modified.
int orc_build(const int64_t* keys, int64_t n, int64_t cap, int n_slots, const int32_t* dims,
              orc_table** out) {
  *out = nullptr;
  if (n < 0 || cap <= n || (cap & (cap - 1)) != 0 || n_slots < 1 || n_slots > 65535) return ORC_INVALID;
  orc_table* t = new orc_table();
  t->n = n;
  t->cap = cap;
  t->n_slots = n_slots;
  t->dims.assign(dims, dims + n_slots);
  t->keys.assign(keys, keys + n);
  t->row_of.reserve((size_t)n);
  t->elem_off.resize((size_t)n + 1);
  t->elem_off[0] = 0;
  for (int64_t i = 0; i < n; ++i) {
    int64_t k = keys[i];
    if (k == kEmpty) { delete t; return ORC_RESERVED_KEY; }
    int s = slot_of_key(k);
    if (s >= n_slots) { delete t; return ORC_BAD_SLOT; }
    if (!t->row_of.emplace(k, i).second) { delete t; return ORC_DUP_KEY; }
    t->elem_off[i + 1] = t->elem_off[i] + dims[s];
  }
  // Linear probing: start at fmix64(key) mod cap, step +1 (wrapping) to the
  // first empty slot.
  const uint64_t mask = (uint64_t)cap - 1;
  t->slot_key.assign((size_t)cap, kEmpty);
  t->slot_row.assign((size_t)cap, -1);
  for (int64_t i = 0; i < n; ++i) {
    uint64_t h = fmix64((uint64_t)keys[i]) & mask;
    int64_t len = 1;
    while (t->slot_key[h] != kEmpty) {
      h = (h + 1) & mask;
      ++len;
    }
    t->slot_key[h] = keys[i];
    t->slot_row[h] = i;
    t->sum_probe += len;
    if (len > t->max_probe) t->max_probe = len;
  }
  // Longest cyclic run of occupied slots; start the scan just after an empty slot.
  if (n > 0) {
    int64_t e = 0;
    while (t->slot_key[e] != kEmpty) ++e;
    int64_t run = 0;
    for (int64_t j = 1; j <= cap; ++j) {
      int64_t p = (e + j) & (int64_t)mask;
      if (t->slot_key[p] != kEmpty) {
        ++run;
        if (run > t->max_cluster) t->max_cluster = run;
      } else {
        run = 0;
      }
    }
  }
  *out = t;
  return ORC_OK;
}

void orc_free(orc_table* t) { delete t; }

// [n, cap, max_probe, sum_probe, max_cluster, n_elems]
int orc_info(const orc_table* t, int64_t* info) {
  info[0] = t->n;
  info[1] = t->cap;
  info[2] = t->max_probe;
  info[3] = t->sum_probe;
  info[4] = t->max_cluster;
  info[5] = t->elem_off[(size_t)t->n];
  return ORC_OK;
}

int orc_layout(const orc_table* t, int64_t* slot_key, int64_t* slot_row) {
  std::memcpy(slot_key, t->slot_key.data(), sizeof(int64_t) * (size_t)t->cap);
  std::memcpy(slot_row, t->slot_row.data(), sizeof(int64_t) * (size_t)t->cap);
  return ORC_OK;
}

int orc_elem_offsets(const orc_table* t, int64_t* off) {
  std::memcpy(off, t->elem_off.data(), sizeof(int64_t) * ((size_t)t->n + 1));
  return ORC_OK;
}

// Resolve query keys two ways: the probe walk over the simulated layout gives
// the slot; the key->row map gives membership and row.  They must agree.
int orc_resolve(const orc_table* t, const int64_t* q, int64_t nq, int64_t* slot_out, int64_t* row_out) {
  const uint64_t mask = (uint64_t)t->cap - 1;
  int rc = ORC_OK;
  for (int64_t i = 0; i < nq; ++i) {
    int64_t k = q[i];
    int64_t slot = -1;
    if (k != kEmpty) {
      uint64_t h = fmix64((uint64_t)k) & mask;
      while (t->slot_key[h] != kEmpty) {
        if (t->slot_key[h] == k) { slot = (int64_t)h; break; }
        h = (h + 1) & mask;
      }
    }
    auto it = t->row_of.find(k);
    int64_t row = (it == t->row_of.end()) ? -1 : it->second;
    if ((slot < 0) != (row < 0) || (slot >= 0 && t->slot_row[slot] != row)) rc = ORC_DISAGREE;
    slot_out[i] = slot;
    row_out[i] = row;
  }
  return rc;
}

namespace {
double load_value(const void* values, int wdtype, int64_t e) {
  if (wdtype == 1) return (double)(float)((const _Float16*)values)[e];
  return (double)((const float*)values)[e];
}
}  // namespace

// EmbeddingBag forward ([JD] 4.2.1): per bag, sequential double sum of the
// rows of the bag's hit keys, then /L for mean.  Writes, for each listed bag
// in list order, dims[slot] doubles of the pooled value and of sum |terms|.
// values: ragged rows in keys-array order, or (row_map != NULL) a compact
// array where row r starts at element row_map[r] (-1: not provided).
int orc_forward(const orc_table* t, const int64_t* offsets, int64_t n_bags, const int64_t* qkeys,
                int pool, int wdtype, const void* values, const int64_t* row_map,
                const int64_t* bag_list, int64_t n_list, double* out, double* absum) {
  if (n_bags % t->n_slots != 0) return ORC_INVALID;
  int64_t count = n_list < 0 ? n_bags : n_list;
  int64_t o = 0;
  for (int64_t li = 0; li < count; ++li) {
    int64_t bag = n_list < 0 ? li : bag_list[li];
    if (bag < 0 || bag >= n_bags) return ORC_INVALID;
    int s = (int)(bag % t->n_slots);
    int D = t->dims[(size_t)s];
    std::vector<double> acc((size_t)D, 0.0), ab((size_t)D, 0.0);
    int64_t L = offsets[bag + 1] - offsets[bag];
    for (int64_t i = offsets[bag]; i < offsets[bag + 1]; ++i) {
      int64_t k = qkeys[i];
      auto it = t->row_of.find(k);
      if (it == t->row_of.end() || slot_of_key(k) != s) continue;  // miss: zero vector
      int64_t r = it->second;
      int64_t e0 = row_map ? row_map[r] : t->elem_off[(size_t)r];
      if (e0 < 0) return ORC_MISSING_ROW;
      for (int j = 0; j < D; ++j) {
        double v = load_value(values, wdtype, e0 + j);
        acc[(size_t)j] += v;
        ab[(size_t)j] += std::fabs(v);
      }
    }
    for (int j = 0; j < D; ++j) {
      double v = acc[(size_t)j], a = ab[(size_t)j];
      if (pool == 1) {
        v = L > 0 ? v / (double)L : 0.0;
        a = L > 0 ? a / (double)L : 0.0;
      }
      out[o + j] = v;
      absum[o + j] = a;
    }
    o += D;
  }
  return ORC_OK;
}

// Backward of the pooled lookup: every hit occurrence of key k in bag
// (b, s) adds grad_out[b, cols of s] (times 1/L for mean) to G[k]; the
// per-key gradient map gives the unique-key set ([TPCG] 计算优化: one
// backward update per key; [JD] 3.2.1: only keys present are touched).
// key_filter (optional) restricts the map to the listed keys.
int orc_backward(const orc_table* t, const int64_t* offsets, int64_t n_bags, const int64_t* qkeys,
                 int pool, const float* grad, const int64_t* key_filter, int64_t n_filter,
                 orc_grad** out) {
  *out = nullptr;
  if (n_bags % t->n_slots != 0) return ORC_INVALID;
  std::vector<int64_t> col((size_t)t->n_slots + 1, 0);
  for (int s = 0; s < t->n_slots; ++s) col[(size_t)s + 1] = col[(size_t)s] + t->dims[(size_t)s];
  const int64_t sumD = col[(size_t)t->n_slots];
  std::unordered_set<int64_t> filter;
  if (key_filter) filter.insert(key_filter, key_filter + n_filter);
  std::map<int64_t, std::pair<std::vector<double>, std::vector<double>>> G;
  for (int64_t bag = 0; bag < n_bags; ++bag) {
    int64_t b = bag / t->n_slots;
    int s = (int)(bag % t->n_slots);
    int D = t->dims[(size_t)s];
    int64_t L = offsets[bag + 1] - offsets[bag];
    double scale = (pool == 1) ? 1.0 / (double)L : 1.0;
    const float* g = grad + b * sumD + col[(size_t)s];
    for (int64_t i = offsets[bag]; i < offsets[bag + 1]; ++i) {
      int64_t k = qkeys[i];
      if (key_filter && !filter.count(k)) continue;
      if (!t->row_of.count(k) || slot_of_key(k) != s) continue;
      auto& e = G[k];
      if (e.first.empty()) {
        e.first.assign((size_t)D, 0.0);
        e.second.assign((size_t)D, 0.0);
      }
      for (int j = 0; j < D; ++j) {
        double term = (double)g[j] * scale;
        e.first[(size_t)j] += term;
        e.second[(size_t)j] += std::fabs(term);
      }
    }
  }
  orc_grad* r = new orc_grad();
  r->goff.push_back(0);
  for (auto& kv : G) {
    r->keys.push_back(kv.first);
    r->rows.push_back(t->row_of.at(kv.first));
    r->G.insert(r->G.end(), kv.second.first.begin(), kv.second.first.end());
    r->A.insert(r->A.end(), kv.second.second.begin(), kv.second.second.end());
    r->goff.push_back((int64_t)r->G.size());
  }
  *out = r;
  return ORC_OK;
}

int orc_grad_info(const orc_grad* g, int64_t* n_unique, int64_t* n_elems) {
  *n_unique = (int64_t)g->keys.size();
  *n_elems = (int64_t)g->G.size();
  return ORC_OK;
}

int orc_grad_copy(const orc_grad* g, int64_t* keys, int64_t* rows, int64_t* goff, double* G, double* A) {
  std::memcpy(keys, g->keys.data(), sizeof(int64_t) * g->keys.size());
  std::memcpy(rows, g->rows.data(), sizeof(int64_t) * g->rows.size());
  std::memcpy(goff, g->goff.data(), sizeof(int64_t) * g->goff.size());
  std::memcpy(G, g->G.data(), sizeof(double) * g->G.size());
  std::memcpy(A, g->A.data(), sizeof(double) * g->A.size());
  return ORC_OK;
}

void orc_grad_free(orc_grad* g) { delete g; }

// Element-wise Adagrad ([JD] 3.2.1; [META] 3.3), float32 arithmetic in this
// order per element:  g = (float)G;  a = acc + g*g;  w = w - (lr*g)/(sqrt(a)+eps).
// Half weights are read exactly as float and the result is rounded to half
// (IEEE round-to-nearest-even).  w and acc are updated in place.
int orc_adagrad(const double* G, int64_t n, int wdtype, void* w, float* acc, float lr, float eps) {
  for (int64_t i = 0; i < n; ++i) {
    float g = (float)G[i];
    float gg = g * g;
    float a = acc[i] + gg;
    float wv = (wdtype == 1) ? (float)((_Float16*)w)[i] : ((float*)w)[i];
    float step = lr * g;
    float den = std::sqrt(a) + eps;
    float nw = wv - step / den;
    acc[i] = a;
    if (wdtype == 1)
      ((_Float16*)w)[i] = (_Float16)nw;
    else
      ((float*)w)[i] = nw;
  }
  return ORC_OK;
}

// Row-wise Adagrad: Adagrad ([JD] 3.2.1) with one accumulator per row instead
// of one per element.  The pages give no formula for this variant; the
// reading here adds the mean of the row's squared gradient.  Per row r of D
// elements (rows given by goff), in float32 and this order:
//   g_d = (float)G_d;  s = sum_d g_d*g_d (d ascending);  m = s / D;
//   a = acc[r] + m;  den = sqrt(a) + eps;  w_d = w_d - (lr*g_d)/den.
// Half weights are read exactly and the result rounded to half (RNE).
int orc_rowwise_adagrad(const double* G, const int64_t* goff, int64_t n_rows, int wdtype, void* w, float* acc,
                        float lr, float eps) {
  for (int64_t r = 0; r < n_rows; ++r) {
    const int64_t b = goff[r], e = goff[r + 1];
    if (e <= b) continue;
    float s = 0.f;
    for (int64_t i = b; i < e; ++i) {
      const float g = (float)G[i];
      s = s + g * g;
    }
    const float m = s / (float)(e - b);
    const float a = acc[r] + m;
    const float den = std::sqrt(a) + eps;
    acc[r] = a;
    for (int64_t i = b; i < e; ++i) {
      const float g = (float)G[i];
      const float wv = (wdtype == 1) ? (float)((_Float16*)w)[i] : ((float*)w)[i];
      const float nw = wv - (lr * g) / den;
      if (wdtype == 1)
        ((_Float16*)w)[i] = (_Float16)nw;
      else
        ((float*)w)[i] = nw;
    }
  }
  return ORC_OK;
}

// FTRL-Proximal, per coordinate (McMahan et al., "Ad Click Prediction: a View
// from the Trenches", KDD 2013, Algorithm 1; the JD article 3.2.1 names FTRL as
// the other sparse optimizer of CTR training).  For each element, with the
// weight w the forward used and the state (z, n), float32 arithmetic in this
// order:
//   g = (float)G;  n' = n + g*g;  sigma = (sqrt(n') - sqrt(n)) / alpha;
//   z' = (z + g) - sigma * w;
//   w' = 0 if |z'| <= lambda1, else -((z' - sign(z') lambda1) / ((beta + sqrt(n')) / alpha + lambda2)).
// Half weights are read exactly and the result rounded to half (RNE).
int orc_ftrl(const double* G, int64_t n, int wdtype, void* w, float* nacc, float* z, float alpha, float beta,
             float l1, float l2) {
  for (int64_t i = 0; i < n; ++i) {
    float g = (float)G[i];
    float wv = (wdtype == 1) ? (float)((_Float16*)w)[i] : ((float*)w)[i];
    float n0 = nacc[i];
    float gg = g * g;
    float n1 = n0 + gg;
    float sn = std::sqrt(n0);
    float sn1 = std::sqrt(n1);
    float sigma = (sn1 - sn) / alpha;
    float zs = z[i] + g;
    float sw = sigma * wv;
    float z1 = zs - sw;
    float nw;
    if (std::fabs(z1) <= l1) {
      nw = 0.0f;
    } else {
      float num = z1 - (z1 > 0.0f ? l1 : -l1);
      float den = (beta + sn1) / alpha + l2;
      nw = -(num / den);
    }
    nacc[i] = n1;
    z[i] = z1;
    if (wdtype == 1)
      ((_Float16*)w)[i] = (_Float16)nw;
    else
      ((float*)w)[i] = nw;
  }
  return ORC_OK;
}

// float -> half, IEEE round-to-nearest-even (the oracle's writeback rounding).
int orc_f32_to_f16(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    _Float16 h = (_Float16)x[i];
    std::memcpy(&out[i], &h, 2);
  }
  return ORC_OK;
}

}  // extern "C"
