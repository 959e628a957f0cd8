// Forward: unified lookup + merged pooling (kernel F).
//
// Tencent PCG DataFun talk, "计算优化": one lookup kernel serves every feature
// of the unified table, pooling of all slots is merged into it ("kernel
// merge"), and FP16 rows are read with vector loads.  JD ads article, 4.2.1:
// per-sample bags pooled by sum or mean.
//
// Mapping (one launch for every slot and dim): one team of TEAM lanes (8, 16
// or 32: a warp holds 32/TEAM teams) per bag, grid-stride over bags in CSR
// order.  The team resolves up to TEAM keys of the bag at once (one key per
// lane: their probes are in flight together), then its lanes split into
// P = TEAM/G groups of G lanes; group p pools keys p, p+P, ...
// of the chunk, each lane owning 16-byte column vectors of the row.  U keys
// per group are gathered before any is added, so every lane keeps U x NCB
// 16-byte loads in flight.  The P partial sums are combined with xor
// shuffles and group 0 writes the pooled row with 16-byte stores.
// Accumulation is float32 in a fixed order, so results are deterministic.
#include <algorithm>
#include <cmath>

#include "emb_internal.cuh"

namespace emb {

template <typename TW>
struct VecOf;
template <>
struct VecOf<float> {
  static constexpr int kElems = 4;
  __device__ __forceinline__ static void add(float* acc, const uint4& v) {
    acc[0] += __uint_as_float(v.x);
    acc[1] += __uint_as_float(v.y);
    acc[2] += __uint_as_float(v.z);
    acc[3] += __uint_as_float(v.w);
  }
};
template <>
struct VecOf<__half> {
  static constexpr int kElems = 8;
  __device__ __forceinline__ static void add(float* acc, const uint4& v) {
    const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 f = __half22float2(h);
      acc[2 * i] += f.x;
      acc[2 * i + 1] += f.y;
    }
  }
};

__device__ __forceinline__ uint4 ldg16(const void* p) {
  uint4 v;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void st16_streaming(float* p, float a, float b, float c, float d) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// Eight pooled floats times s, one whole 32-byte sector, in one streaming store.
__device__ __forceinline__ void st32_streaming(float* p, const float* v, float s) {
  asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(v[0] * s), "f"(v[1] * s),
               "f"(v[2] * s), "f"(v[3] * s), "f"(v[4] * s), "f"(v[5] * s), "f"(v[6] * s), "f"(v[7] * s)
               : "memory");
}

__device__ __forceinline__ int pow2_at_least(int x) {
  int g = 1;
  while (g < x) g <<= 1;
  return g;
}

// With a Record sink the kernel also writes, for the backward, the resolved
// internal row of every occurrence (n_rows for a miss) and its bag, plus 1/L
// per bag for mean pooling.  The pairs go to the bag's place in slot-major
// order (dest), so the backward's sort only has to order rows within a slot.
struct Record {
  unsigned* K;
  unsigned* V;
  float* scale;
  const unsigned* dest;      // first position of each bag's pairs, slot-major: dest[s * B + b]
  unsigned long long B;      // samples in the batch
  unsigned long long* work;  // optional bag counter: bags taken in batches, in order
};

constexpr int kBagBatch = 32;  // bags per counter increment

// Bounded to 8 resident blocks (full occupancy): the gathers are latency
// bound, and resident warps beat registers (measured at 100M keys x dim 128).
template <typename TW, int TEAM, int NCB, int U, bool kRecord>
__global__ void __launch_bounds__(256, 8) fwd_pool_kernel(TableView t, const long long* __restrict__ offsets,
                                                       long long n_bags, const long long* __restrict__ keys,
                                                       long long nnz, int mean, float* __restrict__ out, Record rec) {
  constexpr int VEC = VecOf<TW>::kElems;
  constexpr int BPW = 32 / TEAM;  // bags a warp works on side by side
  const int lane = threadIdx.x & 31;
  const int team = lane / TEAM, tl = lane % TEAM;
  const unsigned tmask = TEAM == 32 ? 0xffffffffu : (((1u << TEAM) - 1u) << (team * TEAM));
  const long long nteams = (((long long)gridDim.x * blockDim.x) >> 5) * BPW;
  const TW* W = static_cast<const TW*>(t.W);
  const int G0 = t.uniform_dim ? min(TEAM, pow2_at_least(t.uniform_dim / VEC)) : 0;  // lanes per key, one dim
  // bags: a static grid-stride order, or batches of kBagBatch consecutive bags
  // taken in order from a counter (balances warps over bags of very
  // different lengths)
  long long stat = ((blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5) * BPW + team;
  // CSR offsets (and, recording, the pairs' slot-major positions) of a team's
  // batch of bags, staged in shared memory with one load per lane: each bag
  // then starts its key -> slot -> row chain without two dependent global reads
  __shared__ long long s_off[8][BPW][kBagBatch + 1];
  __shared__ unsigned s_dst[8][BPW][kBagBatch];
  const int wib = threadIdx.x >> 5;
  for (;;) {
    long long b_lo, b_hi;
    if (rec.work) {
      unsigned long long v = 0;
      if (tl == 0) v = atomicAdd(rec.work, (unsigned long long)kBagBatch);
      b_lo = (long long)__shfl_sync(tmask, v, 0, TEAM);  // also: the team is done with the last batch
      b_hi = min(b_lo + kBagBatch, n_bags);
      if (b_lo < n_bags) {
        const int nb = (int)(b_hi - b_lo);
        for (int j = tl; j <= nb; j += TEAM) s_off[wib][team][j] = offsets[b_lo + j];
        if (kRecord)
          for (int j = tl; j < nb; j += TEAM) {
            const unsigned bj = (unsigned)(b_lo + j);
            s_dst[wib][team][j] = rec.dest[(unsigned long long)(bj % (unsigned)t.n_slots) * rec.B +
                                           bj / (unsigned)t.n_slots];
          }
      }
      __syncwarp(tmask);
    } else {
      b_lo = stat;
      b_hi = stat + 1;
      stat += nteams;
    }
    if (b_lo >= n_bags) break;
  for (long long bag = b_lo; bag < b_hi; ++bag) {
    const int s = (int)((unsigned)bag % (unsigned)t.n_slots);
    const long long b = (unsigned)bag / (unsigned)t.n_slots;
    int D, col;
    long long ebase = 0;
    unsigned rbase = 0;
    if (t.uniform_dim) {
      D = t.uniform_dim;
      col = s * D;
    } else {
      const SlotInfo si = t.sinfo[s];
      D = si.dim;
      col = si.col;
      ebase = si.elem_base;
      rbase = si.row_base;
    }
    const int G = t.uniform_dim ? G0 : min(TEAM, pow2_at_least(D / VEC));  // lanes per key
    const int P = TEAM / G;                           // keys pooled side by side
    const int sub = tl / G, li = tl % G;

    long long start, end;
    if (rec.work) {
      start = s_off[wib][team][bag - b_lo];
      end = s_off[wib][team][bag - b_lo + 1];
    } else {
      start = offsets[bag];
      end = offsets[bag + 1];
    }
    if (start < 0 || end > nnz || end < start || (bag == 0 && start != 0) || (bag == n_bags - 1 && end != nnz)) {
      if (tl == 0) atomicOr(t.flags, EMB_FLAG_BAD_OFFSETS);
      start = min(max(start, 0LL), nnz);
      end = min(max(end, start), nnz);
    }
    // where this bag's pairs go (inside [0, nnz) unless the offsets are malformed)
    const long long d0 =
        kRecord ? (long long)(rec.work ? s_dst[wib][team][bag - b_lo]
                                       : rec.dest[(unsigned long long)s * rec.B + (unsigned long long)b]) - start
                : 0;
    float acc[NCB][VEC];
#pragma unroll
    for (int c = 0; c < NCB; ++c)
#pragma unroll
      for (int j = 0; j < VEC; ++j) acc[c][j] = 0.f;

    for (long long c0 = start; c0 < end; c0 += TEAM) {
      const int n = (int)min((long long)TEAM, end - c0);
      long long elem = -1;  // first weight element of this lane's key, -1 = miss
      if (tl < n) {
        const long long k = keys[c0 + tl];
        unsigned row = t.n_rows;
        if (key_slot(k) != s) {
          atomicOr(t.flags, EMB_FLAG_SLOT_MISMATCH);
        } else {
          unsigned r, ext;
          unsigned long long h;
          if (probe(t, k, &r, &ext, &h)) {
            row = r;
            elem = t.uniform_dim ? (long long)r * D : ebase + (long long)(r - rbase) * D;
          }
        }
        if (kRecord) {
          const long long p = d0 + c0 + tl;
          if (p < nnz) {
            rec.K[p] = row;
            rec.V[p] = (unsigned)bag;
          }
        }
      }
      for (int base = 0; base < n; base += P * U) {
        uint4 v[U][NCB];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = base + u * P + sub;
          const long long e = __shfl_sync(tmask, elem, i & (TEAM - 1), TEAM);
          const bool ok = (i < n) && (e >= 0);
#pragma unroll
          for (int c = 0; c < NCB; ++c) {
            const int ce = (c * G + li) * VEC;
            v[u][c] = (ok && ce < D) ? ldg16(W + e + ce) : make_uint4(0u, 0u, 0u, 0u);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int c = 0; c < NCB; ++c) VecOf<TW>::add(acc[c], v[u][c]);
      }
    }
    // combine the P key groups of the team (fixed xor tree: deterministic)
#pragma unroll
    for (int c = 0; c < NCB; ++c)
#pragma unroll
      for (int j = 0; j < VEC; ++j)
        for (int off = G; off < TEAM; off <<= 1) acc[c][j] += __shfl_xor_sync(tmask, acc[c][j], off, TEAM);

    if (kRecord && mean && tl == 0) rec.scale[bag] = end > start ? 1.0f / (float)(end - start) : 0.f;
    if (sub == 0) {
      const long long L = end - start;
      // mean over L counting misses, as one reciprocal times each sum (within
      // one rounding of the quotient); L = 0 gives 0
      const float inv = (mean && L > 0) ? 1.f / (float)L : 1.f;
      float* o = out + b * t.sum_dims + col;
#pragma unroll
      for (int c = 0; c < NCB; ++c) {
        const int ce = (c * G + li) * VEC;
        if (ce < D) {
          // a lane's 8 floats (f16 rows) are one sector: written whole when
          // aligned, so no sector reaches DRAM half-written
          if (VEC == 8 && ((uintptr_t)(o + ce) & 31) == 0) {
            st32_streaming(o + ce, acc[c], inv);
          } else {
#pragma unroll
            for (int j = 0; j < VEC; j += 4)
              st16_streaming(o + ce + j, acc[c][j] * inv, acc[c][j + 1] * inv, acc[c][j + 2] * inv,
                             acc[c][j + 3] * inv);
          }
        }
      }
    }
  }
  }
}

// Lanes per bag: enough for the widest row's 16-byte vectors and for the
// mean bag's keys to be probed at once, at least 8 and at most a warp.
// Measured: 100 slots x dim 32 f16 with 5.5-key bags, 8 lanes 2.32 ms against
// 4.40 ms for a warp per bag; 26 slots x dim 64 f32 with 10.5-key bags, 16
// lanes 0.388 ms against 0.419; the 100M-key workload (33.7-key bags) and
// the ragged one (rows up to 32 vectors) keep a whole warp.
static int fwd_team(int max_vecs, double mean_len) {
  const int want = std::max(max_vecs, (int)std::ceil(mean_len));
  return want <= 8 ? 8 : want <= 16 ? 16 : 32;
}

template <typename TW, bool kRecord>
static cudaError_t launch_fwd(const emb_table* t, const long long* offsets, long long n_bags, const long long* keys,
                              long long nnz, int mean, float* out, Record rec, cudaStream_t st) {
  constexpr int VEC = VecOf<TW>::kElems;
  const int max_vecs = t->st.max_dim / VEC;  // 16-byte vectors in the widest row
  const int team = fwd_team(max_vecs, n_bags > 0 ? (double)nnz / (double)n_bags : 0.0);
  const int ncb = (max_vecs + team - 1) / team;  // column blocks per lane
  const int threads = 256;
  const long long want = std::max(1LL, (n_bags * team + threads - 1) / threads);
  TableView v = t->fwd_view();
  // grid: one wave of resident blocks, grid-stride over bags
#define EMB_FWD(TM, NC, UU)                                                                                 \
  do {                                                                                                      \
    int per_sm = 0;                                                                                         \
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fwd_pool_kernel<TW, TM, NC, UU, kRecord>, threads, 0); \
    const long long blocks = std::min(want, (long long)std::max(1, per_sm) * sm_count());                  \
    fwd_pool_kernel<TW, TM, NC, UU, kRecord><<<(int)blocks, threads, 0, st>>>(v, offsets, n_bags, keys, nnz, mean, \
                                                                               out, rec);                   \
  } while (0)
  if (team == 8) {
    if (ncb <= 1) EMB_FWD(8, 1, 4); else EMB_FWD(8, 2, 2);
  } else if (team == 16) {
    if (ncb <= 1) EMB_FWD(16, 1, 4); else EMB_FWD(16, 2, 2);
  } else {
    // 3 rows in flight per lane: 14.0 ms against 14.9 (4) and 14.5 (2) at
    // 100M keys x dim 128 f16; 0.385 ms against 0.407 (4) at 10M x dim 64 f32
    if (ncb <= 1) EMB_FWD(32, 1, 3);
    else if (ncb <= 2) EMB_FWD(32, 2, 2);
    else EMB_FWD(32, 4, 1);
  }
#undef EMB_FWD
  return cudaGetLastError();
}

// Forward launch, optionally recording (row, bag) pairs for the backward.
cudaError_t launch_forward(const emb_table* t, const long long* offsets, long long n_bags, const long long* keys,
                           long long nnz, int mean, float* out, unsigned* K, unsigned* V, float* scale,
                           const unsigned* dest, unsigned long long* work, cudaStream_t st) {
  const Record rec{K, V, scale, dest, (unsigned long long)n_bags / (unsigned long long)t->st.n_slots, work};
  const bool record = K != nullptr;
  if (t->fwd_half())
    return record ? launch_fwd<__half, true>(t, offsets, n_bags, keys, nnz, mean, out, rec, st)
                  : launch_fwd<__half, false>(t, offsets, n_bags, keys, nnz, mean, out, rec, st);
  return record ? launch_fwd<float, true>(t, offsets, n_bags, keys, nnz, mean, out, rec, st)
                : launch_fwd<float, false>(t, offsets, n_bags, keys, nnz, mean, out, rec, st);
}

emb_status check_batch(const emb_table* t, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                       int64_t nnz, int pool) {
  if (!t) return fail(EMB_ERR_INVALID_ARG, "table is NULL");
  if (n_bags < 0 || nnz < 0) return fail(EMB_ERR_INVALID_ARG, "negative n_bags or nnz");
  if (n_bags > EMB_MAX_BAGS || nnz > EMB_MAX_NNZ) return fail(EMB_ERR_UNSUPPORTED, "batch exceeds EMB_MAX_* limits");
  if (n_bags % t->st.n_slots != 0) return fail(EMB_ERR_INVALID_ARG, "n_bags must be a multiple of n_slots");
  if (!offsets_d || (nnz > 0 && !keys_d)) return fail(EMB_ERR_INVALID_ARG, "offsets or keys is NULL");
  if (pool != EMB_POOL_SUM && pool != EMB_POOL_MEAN) return fail(EMB_ERR_INVALID_ARG, "bad pool mode");
  return EMB_OK;
}

}  // namespace emb

using namespace emb;

extern "C" emb_status emb_lookup_fwd(emb_table* table, const int64_t* offsets_d, int64_t n_bags,
                                     const int64_t* keys_d, int64_t nnz, emb_pool pool, float* out_d,
                                     void* stream) {
  emb_status rc = check_batch(table, offsets_d, n_bags, keys_d, nnz, pool);
  if (rc != EMB_OK) return rc;
  if (n_bags == 0) return EMB_OK;
  if (!out_d) return fail(EMB_ERR_INVALID_ARG, "out is NULL");
  if (((uintptr_t)out_d & 15) != 0) return fail(EMB_ERR_INVALID_ARG, "out must be 16-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = launch_forward(table, (const long long*)offsets_d, n_bags, (const long long*)keys_d, nnz,
                                 pool == EMB_POOL_MEAN, out_d, nullptr, nullptr, nullptr, nullptr, nullptr, st);
  if (e != cudaSuccess) return cuda_fail(e, "fwd_pool_kernel launch");
  return EMB_OK;
}
