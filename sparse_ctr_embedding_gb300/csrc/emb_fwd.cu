// Forward: unified lookup + merged pooling (kernel F).
//
// Tencent PCG DataFun talk, "计算优化": one lookup kernel serves every feature
// of the unified table, pooling of all slots is merged into it ("kernel
// merge"), and FP16 rows are read with vector loads.  JD ads article, 4.2.1:
// per-sample bags pooled by sum or mean.
//
// Mapping (one launch for every slot and dim): one team of TEAM lanes (8, 16
// or 32: a warp holds 32/TEAM teams) per bag.  The plain forward walks the
// bags grid-stride in CSR order; the recording forward takes them 32 at a
// time from a device counter in slot-major order (every sample of slot 0,
// then slot 1, ...), staging the batch's checked CSR bounds and pair
// positions in shared memory.  The team resolves up to TEAM keys of the bag
// at once (one key per lane: their probes are in flight together), then its
// lanes split into P = TEAM/G groups of G lanes; group p pools keys p, p+P,
// ... of the chunk, each lane owning 16-byte column vectors of the row.  U
// keys per group are gathered before any is added, so every lane keeps
// U x NCB 16-byte loads in flight.  The P partial sums are combined with xor
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
  const unsigned* placed;    // nonzero when the bags tile [0, nnz) (else nothing is recorded)
  unsigned long long B;      // samples in the batch
  unsigned long long* work;  // optional bag counter: bags taken in batches, in order
  int slot_major;            // with work: the counter runs over t = s * B + b instead of bag = b * S + s
};

constexpr int kBagBatch = 32;  // bags per counter increment

// Resident 256-thread blocks per SM the register budget is sized for, by team
// width.  The gathers are latency bound, so occupancy and spill-free registers
// trade against each other; measured per team width on the five benchmark
// workloads: 4- and 8-lane teams (100 slots x dim 32 f16) run best at 4 blocks of
// 64 registers (1.74 ms against 2.01 at 8 blocks of 32), 16-lane teams
// (26 slots x dim 64 f32) at 6 (0.320 ms against 0.376), 32-lane teams
// (100M keys x dim 128 f16; the ragged one) at 8 (12.08 ms against 12.17 at
// 6 and 13.95 at 4).
constexpr int fwd_min_blocks(int team) { return team <= 8 ? 4 : team == 16 ? 6 : 8; }
constexpr unsigned kMissRow = 0xFFFFFFFFu;

// Indices are 32-bit: n_bags and nnz are below 2^31 (the boundary checks it),
// so bag numbers, CSR positions and pair positions all fit.
template <typename TW, int TEAM, int NCB, int U, bool kRecord>
__global__ void __launch_bounds__(256, fwd_min_blocks(TEAM)) fwd_pool_kernel(TableView t, const long long* __restrict__ offsets,
                                                                      long long n_bags_l,
                                                                      const long long* __restrict__ keys,
                                                                      long long nnz_l, int mean, float* __restrict__ out,
                                                                      Record rec) {
  constexpr int VEC = VecOf<TW>::kElems;
  constexpr int BPW = 32 / TEAM;  // bags a warp works on side by side
  const unsigned n_bags = (unsigned)n_bags_l, nnz = (unsigned)nnz_l;
  const int lane = threadIdx.x & 31;
  const int team = lane / TEAM, tl = lane % TEAM;
  const unsigned tmask = TEAM == 32 ? 0xffffffffu : (((1u << TEAM) - 1u) << (team * TEAM));
  const unsigned S = (unsigned)t.n_slots;
  const unsigned B = (unsigned)rec.B;
  const bool by_slot = rec.work != nullptr && rec.slot_major != 0;
  const unsigned nteams = ((gridDim.x * blockDim.x) >> 5) * BPW;
  const TW* W = static_cast<const TW*>(t.W);
  const int G0 = t.uniform_dim ? min(TEAM, pow2_at_least(t.uniform_dim / VEC)) : 0;  // lanes per key, one dim
  // bags: a static grid-stride order, or batches of kBagBatch consecutive
  // counter values taken in order (balances warps over bags of very
  // different lengths); a counter value is a bag number, or with by_slot the
  // slot-major number s * B + b of bag b * S + s
  unsigned stat = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * BPW + team;
  // Checked and clamped CSR bounds (start << 32 | end) and, when recording,
  // the pairs' slot-major positions of a team's batch of bags, staged in
  // shared memory by the lanes in parallel: each bag then starts its
  // key -> slot -> row chain without two dependent global reads
  __shared__ unsigned long long s_se[8][BPW][kBagBatch];
  __shared__ unsigned s_dst[8][BPW][kBagBatch];
  const int wib = threadIdx.x >> 5;
  // malformed offsets whose clamped bags do not tile [0, nnz) record nothing
  // (the backward then updates nothing); otherwise every position is in range
  const bool recording = kRecord && *rec.placed != 0;
  for (;;) {
    unsigned b_lo, b_hi;
    if (rec.work) {
      unsigned long long v = 0;
      if (tl == 0) v = atomicAdd(rec.work, (unsigned long long)kBagBatch);
      // below n_bags + 32 x teams < 2^32; also: the team is done with the last batch
      b_lo = (unsigned)__shfl_sync(tmask, v, 0, TEAM);
      b_hi = min(b_lo + (unsigned)kBagBatch, n_bags);
      if (b_lo < n_bags) {
        const int nb = (int)(b_hi - b_lo);
        for (int j = tl; j < nb; j += TEAM) {
          const unsigned tj = b_lo + j;
          unsigned bag = tj;
          if (by_slot) {
            const unsigned ss = tj / B;
            bag = (tj - ss * B) * S + ss;
          }
          long long start = offsets[bag], end = offsets[bag + 1];
          if (start < 0 || end > (long long)nnz || end < start || (bag == 0 && start != 0) ||
              (bag == n_bags - 1 && end != (long long)nnz)) {
            atomicOr(t.flags, EMB_FLAG_BAD_OFFSETS);
            start = min(max(start, 0LL), (long long)nnz);
            end = min(max(end, start), (long long)nnz);
          }
          s_se[wib][team][j] = ((unsigned long long)start << 32) | (unsigned long long)end;
          if (kRecord) s_dst[wib][team][j] = rec.dest[by_slot ? tj : (bag % S) * B + bag / S];
        }
      }
      __syncwarp(tmask);
    } else {
      b_lo = stat;
      b_hi = stat + 1;
      stat += nteams;
    }
    if (b_lo >= n_bags) break;
  for (unsigned tt = b_lo; tt < b_hi; ++tt) {
    unsigned s, b;
    if (by_slot) {
      s = tt / B;
      b = tt - s * B;
    } else {
      b = tt / S;
      s = tt - b * S;
    }
    const unsigned bag = b * S + s;
    int D, col;
    const TW* Wb = W;    // the slot's first row
    unsigned rbase = 0;  // and its internal row number
    if (t.uniform_dim) {
      D = t.uniform_dim;
      col = (int)s * D;
    } else {
      const SlotInfo si = t.sinfo[s];
      D = si.dim;
      col = si.col;
      Wb = W + si.elem_base;
      rbase = si.row_base;
    }
    const int G = t.uniform_dim ? G0 : min(TEAM, pow2_at_least(D / VEC));  // lanes per key
    const int P = TEAM / G;                           // keys pooled side by side
    const int sub = tl / G, li = tl % G;

    unsigned start, end;
    if (rec.work) {  // checked when staged
      const unsigned long long se = s_se[wib][team][tt - b_lo];
      start = (unsigned)(se >> 32);
      end = (unsigned)se;
    } else {
      long long st = offsets[bag], en = offsets[bag + 1];
      if (st < 0 || en > (long long)nnz || en < st || (bag == 0 && st != 0) ||
          (bag == n_bags - 1 && en != (long long)nnz)) {
        if (tl == 0) atomicOr(t.flags, EMB_FLAG_BAD_OFFSETS);
        st = min(max(st, 0LL), (long long)nnz);
        en = min(max(en, st), (long long)nnz);
      }
      start = (unsigned)st;
      end = (unsigned)en;
    }
    // where this bag's pairs go (inside [0, nnz) when recording)
    const unsigned dst = kRecord ? (rec.work ? s_dst[wib][team][tt - b_lo] : rec.dest[s * B + b]) : 0u;
    float acc[NCB][VEC];
#pragma unroll
    for (int c = 0; c < NCB; ++c)
#pragma unroll
      for (int j = 0; j < VEC; ++j) acc[c][j] = 0.f;

    for (unsigned c0 = start; c0 < end; c0 += TEAM) {
      const int n = (int)min((unsigned)TEAM, end - c0);
      unsigned rr = kMissRow;  // row of this lane's key within its slot's rows
      if (tl < n) {
        const long long k = keys[c0 + tl];
        unsigned row = t.n_rows;
        if (key_slot(k) != (int)s) {
          atomicOr(t.flags, EMB_FLAG_SLOT_MISMATCH);
        } else {
          unsigned r, ext;
          unsigned long long h;
          if (probe(t, k, &r, &ext, &h)) {
            row = r;
            rr = r - rbase;
          }
        }
        if (recording) {  // the bags tile [0, nnz): the position is inside it
          const unsigned p = dst + (c0 - start) + tl;
          rec.K[p] = row;
          rec.V[p] = bag;
        }
      }
      for (int base = 0; base < n; base += P * U) {
        uint4 v[U][NCB];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = base + u * P + sub;
          const unsigned ri = __shfl_sync(tmask, rr, i & (TEAM - 1), TEAM);
          const bool ok = (i < n) && (ri != kMissRow);
          const TW* rp = Wb + (size_t)ri * (unsigned)D;
#pragma unroll
          for (int c = 0; c < NCB; ++c) {
            const int ce = (c * G + li) * VEC;
            v[u][c] = (ok && ce < D) ? ldg16(rp + ce) : make_uint4(0u, 0u, 0u, 0u);
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
      const unsigned L = end - start;
      // mean over L counting misses, as one reciprocal times each sum (within
      // one rounding of the quotient); L = 0 gives 0
      const float inv = (mean && L > 0) ? 1.f / (float)L : 1.f;
      float* o = out + (size_t)b * (unsigned)t.sum_dims + col;
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
// mean bag's keys to be probed at once, at least 8 and at most a warp; rows
// of at most 4 vectors on batches of at least 2^20 bags take 4 lanes (a key's
// row is one 4-lane load; enough bags are in flight to hide the probes).
// Measured: 100 slots x dim 32 f16 with 5.5-key bags, 4 lanes 1.53 ms against
// 1.74 with 8 lanes and 4.40 with a warp per bag; 26 slots x dim 64 f32 with
// 10.5-key bags, 16 lanes 0.388 ms against 0.419; the 100M-key workload
// (33.7-key bags) and the ragged one (rows up to 32 vectors) keep a whole
// warp; the 1024-bag workload (rows of 4 vectors) takes 0.127 ms with 8
// lanes against 0.184 with 4.
static int fwd_team(int max_vecs, double mean_len, long long n_bags) {
  if (max_vecs <= 4 && n_bags >= (1LL << 20)) return 4;
  const int want = std::max(max_vecs, (int)std::ceil(mean_len));
  return want <= 8 ? 8 : want <= 16 ? 16 : 32;
}

template <typename TW, bool kRecord>
static cudaError_t launch_fwd(const emb_table* t, const long long* offsets, long long n_bags, const long long* keys,
                              long long nnz, int mean, float* out, Record rec, cudaStream_t st) {
  constexpr int VEC = VecOf<TW>::kElems;
  const int max_vecs = t->st.max_dim / VEC;  // 16-byte vectors in the widest row
  const int team = fwd_team(max_vecs, n_bags > 0 ? (double)nnz / (double)n_bags : 0.0, n_bags);
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
  if (team == 4) {
    EMB_FWD(4, 1, 4);
  } else if (team == 8) {
    if (ncb <= 1) EMB_FWD(8, 1, 4); else EMB_FWD(8, 2, 2);
  } else if (team == 16) {
    if (ncb <= 1) EMB_FWD(16, 1, 4); else EMB_FWD(16, 2, 2);
  } else {
    // 1 row in flight per lane (2 per team): 11.17 ms against 11.22 (2),
    // 12.05 (3) and 13.26 (4) at 100M keys x dim 128 f16; 0.651 ms against
    // 0.671 (2) and 0.699 (3) on the ragged workload (fewer registers live
    // at the 32-register budget: fewer spills)
    if (ncb <= 1) EMB_FWD(32, 1, 1);
    else if (ncb <= 2) EMB_FWD(32, 2, 2);
    else EMB_FWD(32, 4, 1);
  }
#undef EMB_FWD
  return cudaGetLastError();
}

// Forward launch, optionally recording (row, bag) pairs for the backward.
cudaError_t launch_forward(const emb_table* t, const long long* offsets, long long n_bags, const long long* keys,
                           long long nnz, int mean, float* out, unsigned* K, unsigned* V, float* scale,
                           const unsigned* dest, const unsigned* placed, unsigned long long* work, cudaStream_t st) {
  // The recording forward takes bags in slot-major order (all samples of
  // slot 0, then slot 1, ...): the gathers then stay inside one slot's block
  // of rows at a time and the recorded pairs are written in place order.
  // Measured: 12.08 ms against 14.15 in sample-major order at 100M keys x
  // dim 128 f16, 2.01 against 2.21 at 100 slots x dim 32 f16, within 0.01 ms
  // on the smaller workloads.
  const int slot_major = work != nullptr ? 1 : 0;
  const Record rec{K,    V, scale, dest, placed, (unsigned long long)n_bags / (unsigned long long)t->st.n_slots,
                   work, slot_major};
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
                                 pool == EMB_POOL_MEAN, out_d, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                 st);
  if (e != cudaSuccess) return cuda_fail(e, "fwd_pool_kernel launch");
  return EMB_OK;
}
