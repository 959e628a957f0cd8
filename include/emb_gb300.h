/*
 * emb_gb300.h -- C ABI of the GB300 (sm_103a) embedding step over a unified,
 * insert-free GPU hash table.
 *
 * The step, as the pages describe it:
 *  - Tencent PCG DataFun talk (GPU recommendation-training framework),
 *    paragraph "各阶段优化详细介绍": before a PASS is trained, every embedding
 *    vector (and optimizer state) it needs is flashed whole into an embedding
 *    table in GPU memory; that table is a GPU hashtable whose insert
 *    operation is removed, because the table structure is prepared
 *    beforehand and copied to global memory as one block.
 *  - same talk, paragraph "计算优化" (Unified Hash Table): all features share
 *    one huge table; keys are int64 with the real key in the low 48 bits and
 *    the table (slot) id in the high 16 bits; one lookup kernel serves all
 *    features and one backward kernel updates them; pooling of identical
 *    parameters is merged ("kernel merge"); FP16 storage allows vectorised
 *    access and half2 arithmetic.
 *  - JD ads sparse-training article, section 4.2.1: an EmbeddingBag over a
 *    flat id list with per-sample offsets, pooled by sum or mean; section
 *    3.2.1: Adagrad keeps a per-parameter sum of squared gradients, updates
 *    element-wise, and leaves features absent from the batch untouched.
 * The hash (MurmurHash3 fmix64), linear probing over a power-of-two table and
 * the update  acc += g*g; w -= lr*g/(sqrt(acc)+eps)  complete the method.
 *
 * Conventions shared by every entry point:
 *  - Pointers named *_h are host memory; *_d are device memory of the GPU
 *    that is current when the call is made.  Arguments documented as "host
 *    or device" accept either (unified addressing).
 *  - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *    default stream.  Calls that take a stream only enqueue work and return;
 *    kernel-side problems are reported later by emb_check_device_flag().
 *  - Every call returns an emb_status and never aborts the process; on
 *    failure emb_last_error() gives a human-readable reason (thread-local).
 *  - The table owns all of its device memory (slots, weights, accumulators);
 *    the caller owns every input, output and workspace buffer.
 *  - Keys: key = (slot << 48) | raw, 0 <= slot < n_slots <= 65535.  The
 *    all-ones int64 (-1) is the empty-slot sentinel and is never a key.
 *  - A CSR batch over B samples and S slots has n_bags = B*S bags in
 *    sample-major order (bag = b*S + s), offsets int64[n_bags+1] with
 *    offsets[0] = 0, nondecreasing, offsets[n_bags] = nnz, and keys
 *    int64[nnz].  Bag (b, s) pools only table keys whose slot field is s;
 *    keys absent from the table (misses) pool as zero vectors.
 *  - Pooled output and its gradient are float32 [B, sum(dims)], slot s
 *    occupying columns [col_s, col_s + dim_s) with col_s = sum_{s'<s} dim_s'.
 */
#ifndef EMB_GB300_H
#define EMB_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define EMB_API __attribute__((visibility("default")))
#else
#define EMB_API
#endif

typedef struct emb_table emb_table; /* opaque; owns the table's device memory */

typedef enum {
  EMB_OK = 0,
  EMB_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad enum, bad layout */
  EMB_ERR_CUDA = 2,         /* a CUDA runtime call failed */
  EMB_ERR_OOM = 3,          /* device or host allocation failed */
  EMB_ERR_DUP_KEY = 4,      /* a key appears twice in emb_table_create */
  EMB_ERR_RESERVED_KEY = 5, /* the empty sentinel (-1) given as a key */
  EMB_ERR_LOAD_FACTOR = 6,  /* capacity not a power of two >= 2 * n_keys */
  EMB_ERR_WORKSPACE = 7,    /* workspace missing or smaller than required */
  EMB_ERR_DEVICE_FLAG = 8,  /* a kernel reported bad input (see flag bits) */
  EMB_ERR_UNSUPPORTED = 9   /* a size beyond this library's stated limits */
} emb_status;

/* Weight storage; the accumulator is always f32.
 *   EMB_F32, EMB_F16: one copy of every row, read by the forward and updated
 *     in place (f16 rows are updated in f32 and rounded to nearest-even).
 *   EMB_F16_MASTER: mixed precision as the JD article describes it (3.2.3:
 *     rows stored and used in FP16, an FP32 copy of the weights kept for the
 *     update): an f32 master row, which the update works on and which is what
 *     create takes and export returns, and an f16 copy of it, which the
 *     forward reads.  After each update the f16 copy of every updated row is
 *     its master rounded to nearest-even.  10 bytes per element with the
 *     accumulator. */
typedef enum { EMB_F32 = 0, EMB_F16 = 1, EMB_F16_MASTER = 2 } emb_dtype;

/* The sparse optimizer a table is created for (JD ads article 3.2.1 names
 * Adagrad and FTRL).  Adagrad keeps one f32 accumulator per element; row-wise
 * Adagrad keeps one f32 accumulator per row (key) and adds the mean of the
 * row's squared gradient to it (the pages give no formula for this variant;
 * this is the reading); FTRL keeps two f32 state values per element, n (in
 * the accumulator array) and z.  The Adagrad entry points apply the rule of
 * the table (element-wise or row-wise); a backward call of the other
 * optimizer family is refused.  Accumulator arrays (emb_table_create's acc,
 * emb_table_export's acc_out, emb_table_export_rows' acc_out_d) hold one
 * value per element, or per key for row-wise tables. */
typedef enum { EMB_OPT_ADAGRAD = 0, EMB_OPT_FTRL = 1, EMB_OPT_ROWWISE_ADAGRAD = 2 } emb_optimizer;
typedef enum { EMB_POOL_SUM = 0, EMB_POOL_MEAN = 1 } emb_pool;

/* Device flag bits reported by emb_check_device_flag. */
#define EMB_FLAG_PROBE_BOUND 1u   /* a probe ran past the table's longest cluster (corrupt table) */
#define EMB_FLAG_BAD_OFFSETS 2u   /* CSR offsets out of [0, nnz] or decreasing; clamped */
#define EMB_FLAG_SLOT_MISMATCH 4u /* a bag held a key of another slot; it was skipped */
#define EMB_FLAG_BAD_ROW 8u       /* emb_table_export_rows got a row index outside [0, n_keys) */

/* Limits of this implementation (EMB_ERR_UNSUPPORTED beyond them). */
#define EMB_MAX_DIM 512            /* per-slot dim; f32 dims multiple of 4, f16 of 8 */
#define EMB_MAX_KEYS 2147483647LL  /* rows are indexed with 32 bits */
#define EMB_MAX_NNZ 2147483647LL   /* per call */
#define EMB_MAX_BAGS 2147483647LL  /* per call */

/* Digit width of the backward's stable radix sort of (row, bag) pairs.  The
 * pairs are placed slot by slot, so only the row number within a slot is
 * sorted: ceil(bits(max_slot_keys) / EMB_SORT_DIGIT_BITS) passes (at least
 * one), each one digit-count, three scan and one scatter launch (no
 * counterpart in the pages; stated so callers can count the kernels a step
 * launches). */
#define EMB_SORT_DIGIT_BITS 7

typedef struct {
  int32_t n_slots;         /* feature tables merged into the unified table, 1..65535 */
  const int32_t* slot_dim; /* host [n_slots]: embedding dim of each slot */
  emb_dtype wdtype;        /* weight storage type */
  int64_t capacity;        /* slots: power of two >= 2*n_keys; 0 = the smallest such */
  float acc_init;          /* accumulator (FTRL: n) value used when emb_table_create gets acc == NULL */
  emb_optimizer optimizer; /* EMB_OPT_ADAGRAD (0), EMB_OPT_FTRL (FTRL tables start with z = 0) or
                              EMB_OPT_ROWWISE_ADAGRAD */
} emb_table_desc;

/* FTRL-Proximal hyperparameters (McMahan et al., KDD 2013): alpha > 0,
 * beta, lambda1, lambda2 >= 0. */
typedef struct {
  float alpha;
  float beta;
  float lambda1;
  float lambda2;
} emb_ftrl_params;

typedef struct {
  int64_t n_keys;
  int64_t capacity;
  int64_t n_elems;     /* weight elements = sum over keys of dim(slot(key)) */
  int32_t n_slots;
  int32_t sum_dims;    /* columns of the pooled output */
  int32_t max_dim;
  int32_t wdtype;
  int64_t max_probe;   /* longest probe sequence (slots inspected) of an inserted key */
  int64_t sum_probe;   /* sum over inserted keys of their probe lengths */
  int64_t max_cluster; /* longest run of occupied slots */
  int64_t probe_bound; /* max_cluster + 1: kernels never inspect more slots per key */
  double load_factor;  /* n_keys / capacity */
  uint64_t device_bytes;
  int64_t max_slot_keys; /* keys of the largest slot (the backward sorts rows within a slot) */
} emb_table_stats;

/*
 * emb_table_create -- prepare the insert-free table and flash it to the GPU
 * (Tencent PCG talk, "各阶段优化详细介绍"; key layout from "计算优化").
 *   desc     host: slot count, per-slot dims, weight type, capacity, acc_init.
 *   keys_h   host int64[n_keys]: the deduplicated keys of the pass, in
 *            "keys-array order".  Slots are assigned by inserting the keys one
 *            by one in this order with linear probing from fmix64(key) mod
 *            capacity, so the layout is a pure function of this array.
 *   values   host or device, ragged rows in keys-array order: key i's row has
 *            dim(slot(key_i)) elements of wdtype (float, IEEE half, or float
 *            for EMB_F16_MASTER: the master rows, whose f16 copy is made
 *            here).  NULL fills the weights with zeros.
 *   acc      host or device float32, same element layout as values (row-wise
 *            tables: one value per key, in keys-array order); NULL fills
 *            with desc->acc_init.
 *   stream   stream for the uploads; the call synchronises it before return.
 *   out      receives the table handle (NULL on failure).
 * Errors: INVALID_ARG (bad desc, slot field >= n_slots, dims out of range),
 * RESERVED_KEY, DUP_KEY, LOAD_FACTOR, UNSUPPORTED (n_keys > EMB_MAX_KEYS),
 * OOM, CUDA.  Nothing is left allocated on failure.
 */
EMB_API emb_status emb_table_create(const emb_table_desc* desc, const int64_t* keys_h, int64_t n_keys,
                            const void* values, const float* acc, void* stream, emb_table** out);

/*
 * emb_table_create_device -- the same table as emb_table_create, prepared on
 * the GPU from keys already in device memory (Tencent PCG talk,
 * "各阶段优化详细介绍": the table is prepared before the pass and flashed to
 * GPU memory whole; here the preparation itself runs on the GPU).  The slot
 * layout, row numbering, statistics and errors are exactly those of
 * emb_table_create on the same keys: keys inserted in keys-array order with
 * linear probing, reproduced in parallel (sort by home, prefix-max scan of
 * the first-come-first-served positions, then each run of occupied slots
 * replayed in keys-array order).
 *   keys_d   device int64[n_keys]; values and acc as emb_table_create.
 * Limits: capacity <= 2^32, and no run of occupied slots longer than 4096
 * (EMB_ERR_UNSUPPORTED otherwise; at load factor 0.5 runs are a few keys
 * long, only adversarial keys make long ones).  Scratch of about 48 bytes per
 * key is allocated and freed during the call.  Synchronises `stream`.
 */
EMB_API emb_status emb_table_create_device(const emb_table_desc* desc, const int64_t* keys_d, int64_t n_keys,
                                           const void* values, const float* acc, void* stream, emb_table** out);

/* Free the table and its device memory (the end of a pass, Tencent PCG talk,
 * "各阶段优化详细介绍").  Work queued on it must be complete. */
EMB_API emb_status emb_table_destroy(emb_table* table);

/* Host-side statistics of the table (no GPU access): probe lengths and the
 * longest cluster of occupied slots.  The JD ads article (4.3) asks that hash
 * collisions be monitored; this table stores the keys, so two ids never share
 * a row, and what collisions cost here is longer probes, which these count. */
EMB_API emb_status emb_table_get_stats(const emb_table* table, emb_table_stats* out);

/*
 * emb_table_plan -- the preparation step of emb_table_create alone (Tencent
 * PCG talk, "各阶段优化详细介绍": the table structure is prepared before it
 * is flashed to the GPU): validate desc and keys and compute the statistics the
 * table would have, on the host only (no CUDA call).  Same errors as
 * emb_table_create apart from OOM/CUDA.  slot_key_h / slot_row_h, if not
 * NULL, receive the host-built layout: int64[capacity] key per slot (-1 =
 * empty) and the keys-array index stored there (-1 = empty).
 */
EMB_API emb_status emb_table_plan(const emb_table_desc* desc, const int64_t* keys_h, int64_t n_keys,
                          emb_table_stats* out, int64_t* slot_key_h, int64_t* slot_row_h);

/*
 * emb_lookup_fwd -- the unified lookup kernel plus merged pooling (Tencent
 * PCG talk, "计算优化"; JD article 4.2.1): for every bag, probe each key,
 * gather the rows of the hits and sum them in float32; mean divides by the
 * bag length L counting misses (L = 0 gives zeros).
 *   offsets_d  int64[n_bags+1] CSR offsets; n_bags must be a multiple of n_slots.
 *   keys_d     int64[nnz].
 *   out_d      float32[n_bags/n_slots, sum_dims], fully overwritten; 16-byte
 *              aligned (rows are written with 16-byte stores).
 * Errors (host, before any work): INVALID_ARG (also for a misaligned out_d),
 * UNSUPPORTED.  Offsets outside
 * [0, nnz] are clamped and raise EMB_FLAG_BAD_OFFSETS; a key of another slot
 * is skipped and raises EMB_FLAG_SLOT_MISMATCH.
 */
EMB_API emb_status emb_lookup_fwd(emb_table* table, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                          int64_t nnz, emb_pool pool, float* out_d, void* stream);

/* Bytes of device workspace emb_bwd_adagrad needs for this batch shape (no
 * counterpart in the pages: the caller owns the backward's scratch memory). */
EMB_API emb_status emb_bwd_workspace_size(const emb_table* table, int64_t n_bags, int64_t nnz, size_t* bytes);

/*
 * emb_bwd_adagrad -- the unified backward kernel (Tencent PCG talk, "计算优化")
 * with element-wise sparse Adagrad (JD article 3.2.1): every hit occurrence of
 * key k in bag (b, s) contributes grad_out[b, cols of s] (times 1/L for mean)
 * to G[k]; the contributions of duplicate keys are reduced deterministically
 * (stable sort by row, fixed-order segmented sums); then for each hit key and
 * each element:  acc += g*g;  w -= lr*g / (sqrt(acc) + eps)  in float32
 * (half weights rounded to nearest-even).  On a row-wise table (one
 * accumulator a per row of D elements):  a += (sum of g*g over the row) / D;
 * then for each element  w -= lr*g / (sqrt(a) + eps).  Rows not hit are not
 * touched.
 *   grad_out_d   float32[n_bags/n_slots, sum_dims], 16-byte aligned (read with
 *                16-byte vector loads; INVALID_ARG otherwise).
 *   workspace_d  device scratch of at least emb_bwd_workspace_size() bytes,
 *                256-byte aligned; after the call it holds the unique rows of
 *                this step (read them with emb_bwd_unique_keys).
 * Same input checks as emb_lookup_fwd, plus WORKSPACE.  Two calls that share
 * a workspace or a table must be ordered on the GPU (same stream or events).
 */
EMB_API emb_status emb_bwd_adagrad(emb_table* table, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                           int64_t nnz, emb_pool pool, const float* grad_out_d, float lr, float eps,
                           void* workspace_d, size_t ws_bytes, void* stream);

/*
 * emb_bwd_ftrl -- the same backward with the FTRL-Proximal update instead of
 * Adagrad (JD ads article 3.2.1 names FTRL beside Adagrad as the sparse
 * optimizers of CTR training; the update is the per-coordinate form of
 * McMahan et al., "Ad Click Prediction: a View from the Trenches", KDD 2013,
 * Algorithm 1).  For each hit key and each element, with g its summed
 * gradient and w the weight the forward read, in float32:
 *   sigma = (sqrt(n + g*g) - sqrt(n)) / alpha;  z += g - sigma * w;  n += g*g;
 *   w = 0 if |z| <= lambda1, else -(z - sign(z) lambda1) / ((beta + sqrt(n)) / alpha + lambda2)
 * (half weights rounded to nearest-even; master-copy tables update the f32
 * masters).  Rows not hit are not touched.  The table must have been created
 * with optimizer EMB_OPT_FTRL (else EMB_ERR_INVALID_ARG); params is host
 * memory, checked before any work is queued.  Other arguments, errors and
 * ordering rules as emb_bwd_adagrad.
 */
EMB_API emb_status emb_bwd_ftrl(emb_table* table, const int64_t* offsets_d, int64_t n_bags, const int64_t* keys_d,
                                int64_t nnz, emb_pool pool, const float* grad_out_d, const emb_ftrl_params* params,
                                void* workspace_d, size_t ws_bytes, void* stream);

/*
 * emb_bwd_phase_events -- optional timing hook (no counterpart in the pages;
 * it serves measurement).  Registers up to EMB_BWD_PHASES caller-owned
 * cudaEvent_t handles (passed as void*, created with timing enabled) that
 * every later backward call on this table (emb_bwd_adagrad, emb_bwd_ftrl and
 * their recorded and no-alloc forms) records, on its stream, after each of
 * its phases: [0] expand (probe to row/bag pairs; nothing after a recording
 * forward), [1] radix sort, [2] segmented reduce + update, [3] the fold of
 * long rows' partials (large batches) and the cross-chunk fixup.  Elapsed times
 * between an event recorded just before the call and these give each
 * phase's device time.  n = 0 removes the hook.  The events must outlive
 * the calls that record them.
 */
#define EMB_BWD_PHASES 4
EMB_API emb_status emb_bwd_phase_events(emb_table* table, void* const* events, int n);

/*
 * emb_bwd_adagrad_noalloc -- the same backward + Adagrad step as
 * emb_bwd_adagrad, for callers that cannot allocate device memory: code that
 * runs under a memory manager which already owns all of the GPU's memory
 * (for example another framework's caching allocator), or a latency-critical
 * loop whose rules forbid allocation during a step.  The pages have no
 * counterpart of this entry point; it exists only for such callers.
 * Instead of a caller workspace it uses one scratch array that the library
 * holds in device memory, EMB_NOALLOC_SCRATCH_BYTES long, on every GPU that
 * loads the library, until the process exits.  The call allocates nothing.
 *   - A batch whose workspace (emb_bwd_workspace_size) exceeds
 *     EMB_NOALLOC_SCRATCH_BYTES is rejected with EMB_ERR_UNSUPPORTED before
 *     any work is queued (about 3 million lookups fit at dim 128).
 *   - The first call in each CUDA context (per device, and again after a
 *     cudaDeviceReset) looks up the array's device address with
 *     cudaGetSymbolAddress, with that device current, and keeps it for that
 *     context; make that first call before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind.  Calls that can overlap on the GPU (different streams without
 *     ordering, or several threads) race on it and give wrong results: order
 *     them.  No part of the array has to start at zero; each call writes
 *     every region before reading it (with malformed offsets too: positions
 *     outside every bag are written as absent pairs).
 *   - emb_bwd_unique_keys cannot read this array; use emb_bwd_adagrad with a
 *     workspace when the unique keys are needed.
 * Arguments and errors otherwise as emb_bwd_adagrad.
 */
#define EMB_NOALLOC_SCRATCH_BYTES (64u << 20)
EMB_API emb_status emb_bwd_adagrad_noalloc(emb_table* table, const int64_t* offsets_d, int64_t n_bags,
                                           const int64_t* keys_d, int64_t nnz, emb_pool pool,
                                           const float* grad_out_d, float lr, float eps, void* stream);

/*
 * emb_lookup_fwd_record / emb_bwd_adagrad_recorded -- the same forward and
 * backward split so that the probe runs once per step: the lookup kernel of
 * the forward ([TPCG] 计算优化: one kernel resolves every feature) also writes
 * each occurrence's resolved row and bag into `workspace_d` (sized by
 * emb_bwd_workspace_size), and the backward then starts from those pairs
 * instead of probing the keys again.  Output, pooling and update are exactly
 * those of emb_lookup_fwd and emb_bwd_adagrad.
 *   emb_lookup_fwd_record: arguments of emb_lookup_fwd plus the workspace.
 *   emb_bwd_adagrad_recorded: the batch shape (n_bags, nnz, pool) must be the
 *   one recorded last on this table into this same workspace, and the call
 *   must be ordered after the recording forward on the GPU; otherwise it
 *   returns EMB_ERR_INVALID_ARG without queuing work.  The recorded pairs
 *   reflect the keys as the forward read them.
 */
EMB_API emb_status emb_lookup_fwd_record(emb_table* table, const int64_t* offsets_d, int64_t n_bags,
                                         const int64_t* keys_d, int64_t nnz, emb_pool pool, float* out_d,
                                         void* workspace_d, size_t ws_bytes, void* stream);
EMB_API emb_status emb_bwd_adagrad_recorded(emb_table* table, int64_t n_bags, int64_t nnz, emb_pool pool,
                                            const float* grad_out_d, float lr, float eps, void* workspace_d,
                                            size_t ws_bytes, void* stream);
/* The recorded backward with the FTRL update of emb_bwd_ftrl. */
EMB_API emb_status emb_bwd_ftrl_recorded(emb_table* table, int64_t n_bags, int64_t nnz, emb_pool pool,
                                         const float* grad_out_d, const emb_ftrl_params* params, void* workspace_d,
                                         size_t ws_bytes, void* stream);

/*
 * emb_lookup_fwd_dedup -- the forward with a within-batch dedupe (Tencent PCG
 * talk, "各阶段优化详细介绍": a group's keys are deduplicated before their
 * rows are moved): every occurrence is resolved and its (row, bag) pair
 * placed and sorted by row, as the backward does; each unique row is then
 * read from the table once and added into every bag that holds it.  The
 * sorted pairs stay in the workspace, so emb_bwd_adagrad_recorded /
 * emb_bwd_ftrl_recorded called next skip their sort.  Arguments, workspace
 * and errors as emb_lookup_fwd_record.  The pooled adds of a bag come from
 * several warps, as float32 atomics, so `out` agrees with emb_lookup_fwd to
 * within float32 rounding of the sum but is not bitwise reproducible (the
 * update that follows is, as after emb_lookup_fwd_record).
 */
EMB_API emb_status emb_lookup_fwd_dedup(emb_table* table, const int64_t* offsets_d, int64_t n_bags,
                                        const int64_t* keys_d, int64_t nnz, emb_pool pool, float* out_d,
                                        void* workspace_d, size_t ws_bytes, void* stream);

/*
 * emb_bwd_unique_keys -- the deduplicated key set of the last emb_bwd_adagrad
 * that used this workspace (Tencent PCG talk, "各阶段优化详细介绍": the
 * deduplicated keys a group uses are what the pass moves between the GPU table
 * and the slower tiers; here, the keys the step updated).  keys_out_d int64[>= nnz of that call] receives
 * the unique hit keys (slot-major internal row order); n_unique_d int64[1]
 * receives their count.
 */
EMB_API emb_status emb_bwd_unique_keys(const emb_table* table, const void* workspace_d, size_t ws_bytes,
                               int64_t* keys_out_d, int64_t* n_unique_d, void* stream);

/*
 * emb_resolve -- the probe of the unified lookup kernel alone (Tencent PCG
 * talk, "计算优化": one lookup over the unified table resolves every
 * feature's keys), for checking slot resolution: for each key,
 * slot_out_d[i] = its slot index in the table or -1, row_out_d[i] = its index
 * in the keys array given to emb_table_create or -1.  Either output may be NULL.
 */
EMB_API emb_status emb_resolve(const emb_table* table, const int64_t* keys_d, int64_t n, int64_t* slot_out_d,
                       int64_t* row_out_d, void* stream);

/*
 * emb_table_export -- checkpoint (Tencent PCG talk, after "计算优化": a full
 * model is exported every day and an incremental one every hour): copy keys,
 * weights and accumulators back in keys-array order (same layouts as emb_table_create's inputs; the f32 master
 * rows for EMB_F16_MASTER).  Destinations
 * are host or device; any may be NULL.  Synchronises `stream`.  Creating a
 * table from the exported arrays resumes it exactly.
 */
EMB_API emb_status emb_table_export(const emb_table* table, int64_t* keys_out, void* values_out, float* acc_out,
                            void* stream);

/*
 * emb_table_export_rows -- partial checkpoint, the incremental export of the
 * same passage (the rows a step updated, e.g. from emb_bwd_unique_keys): the
 * weights and accumulators of selected keys-array rows (ext_rows_d int64[n], indices into the keys array
 * given at creation).  Outputs are device buffers laid out [n, max_dim]: row
 * i's dim(slot) elements first, zero padding after (the accumulators of a
 * row-wise table: [n], one per row).  Either output may be
 * NULL.  An index outside [0, n_keys) yields a zero row and raises
 * EMB_FLAG_BAD_ROW.  Enqueued on `stream`.
 */
EMB_API emb_status emb_table_export_rows(const emb_table* table, const int64_t* ext_rows_d, int64_t n,
                                         void* values_out_d, float* acc_out_d, void* stream);

/*
 * emb_table_export_z / emb_table_import_z -- the FTRL state z of every
 * element, f32 in keys-array order (the layout of emb_table_create's acc),
 * host or device; the checkpoint and the resume of an FTRL table together
 * with emb_table_export (whose accumulators are FTRL's n).  Synchronise
 * `stream`.  EMB_ERR_INVALID_ARG on a table created for Adagrad.
 */
EMB_API emb_status emb_table_export_z(const emb_table* table, float* z_out, void* stream);
EMB_API emb_status emb_table_import_z(emb_table* table, const float* z_in, void* stream);

/* Copy the slot layout (key and keys-array index per slot, -1 = empty) to
 * host or device int64[capacity] buffers; either may be NULL.  Synchronises.
 * No counterpart in the pages: it exposes the prepared layout for checking. */
EMB_API emb_status emb_table_slots(const emb_table* table, int64_t* slot_key_out, int64_t* slot_row_out, void* stream);

/*
 * emb_check_device_flag -- (no counterpart in the pages: kernels report bad
 * input through a flag word instead of trapping) synchronise `stream`, read
 * and clear the table's device flag word.  Returns EMB_ERR_DEVICE_FLAG if any EMB_FLAG_* bit was set
 * by a kernel since the last check (flags_out, if not NULL, receives them).
 */
EMB_API emb_status emb_check_device_flag(emb_table* table, void* stream, uint32_t* flags_out);

/*
 * Batch pipeline (Tencent PCG talk, "GPU 训练整体架构": the stages of the
 * training step run concurrently as a multi-stage pipeline; JD ads article
 * 3.2.2: sparse updates pipelined with data movement).  The pipeline owns
 * `depth` buffer sets (CSR batch, optionally grad_out, pooled output,
 * backward workspace), an upload stream and a download stream; the step runs
 * on the caller's compute stream.  Per batch, in this order:
 *   emb_pipeline_submit    copy the host CSR batch (and grad_out, if the
 *                          pipeline uploads gradients) into a free set on the
 *                          upload stream; returns a ticket (0, 1, 2, ...).
 *                          It may run ahead of the step by up to depth - 1
 *                          batches: that is the overlap.  A set's inputs are
 *                          overwritten only after its previous batch's
 *                          backward is done (the upload stream waits on the
 *                          GPU; the host does not block).
 *   emb_pipeline_forward   the recording forward of that batch on the compute
 *                          stream, after its upload and after the download of
 *                          the set's previous batch; pooled output into out_d
 *                          (or, NULL, the set's own buffer, returned through
 *                          out_used) and, if out_h is given, copied to out_h
 *                          on the download stream.  A caller's out_d must not
 *                          be written again before that copy is done.
 *   emb_pipeline_backward_adagrad / _ftrl
 *                          the recorded backward of that batch with grad_out_d
 *                          (device) or, NULL, the uploaded grad_out (uploaded
 *                          after the CSR batch, so the forward does not wait
 *                          for it; the backward does); then the set is
 *                          released.  Must come before the next
 *                          batch's forward (the table keeps one recording).
 *   emb_pipeline_release   instead of a backward: release a forwarded set
 *                          (forward-only use).
 *   emb_pipeline_wait      block the host until the batch's backward (or
 *                          release) and download are done (then out_h holds
 *                          its pooled output).
 * Updates are ordered before the next batch's forward, so a pipelined run
 * gives exactly the results of the same calls made one after the other.
 * Host buffers should be pinned for the copies to overlap (pageable memory
 * still works, synchronously).  Not thread-safe: one host thread drives a
 * pipeline.  Errors: INVALID_ARG (bad sizes, tickets out of order, a set
 * still held), OOM / CUDA from create.
 */
typedef struct emb_pipeline emb_pipeline;
EMB_API emb_status emb_pipeline_create(emb_table* table, int64_t max_bags, int64_t max_nnz, int depth,
                                       int upload_grad, void* compute_stream, emb_pipeline** out);
EMB_API emb_status emb_pipeline_destroy(emb_pipeline* pipe);
EMB_API emb_status emb_pipeline_submit(emb_pipeline* pipe, const int64_t* offsets_h, int64_t n_bags,
                                       const int64_t* keys_h, int64_t nnz, const float* grad_out_h,
                                       int64_t* ticket_out);
EMB_API emb_status emb_pipeline_forward(emb_pipeline* pipe, int64_t ticket, emb_pool pool, float* out_d,
                                        float* out_h, float** out_used);
EMB_API emb_status emb_pipeline_backward_adagrad(emb_pipeline* pipe, int64_t ticket, const float* grad_out_d,
                                                 float lr, float eps);
EMB_API emb_status emb_pipeline_backward_ftrl(emb_pipeline* pipe, int64_t ticket, const float* grad_out_d,
                                              const emb_ftrl_params* params);
EMB_API emb_status emb_pipeline_release(emb_pipeline* pipe, int64_t ticket);
EMB_API emb_status emb_pipeline_wait(emb_pipeline* pipe, int64_t ticket);

/*
 * Fault injection, for tests of the failure paths (no counterpart in the
 * pages; everything is injected on the host, no kernel is made to fault).
 *  - emb_debug_fail_device_alloc(after): the next `after` device allocations
 *    of the library succeed and every one after them fails as out of memory,
 *    until called again with a negative value (never fail, the default).
 *    Process-wide.
 *  - emb_debug_live_device_allocs(): device allocations of the library not
 *    yet freed (every table holds some; a failed create leaves none).
 *  - emb_debug_set_probe_bound(table, bound): lower the table's probe bound,
 *    1 <= bound <= max_cluster + 1, as a corrupted table would have it: a key
 *    further than `bound` slots from its home then misses and raises
 *    EMB_FLAG_PROBE_BOUND, and no probe inspects more than `bound` slots.
 */
EMB_API emb_status emb_debug_fail_device_alloc(int64_t after);
EMB_API int64_t emb_debug_live_device_allocs(void);
EMB_API emb_status emb_debug_set_probe_bound(emb_table* table, int64_t bound);

/* Human-readable status name, and the calling thread's last error message
 * (no counterpart in the pages). */
EMB_API const char* emb_status_string(emb_status s);
EMB_API const char* emb_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* EMB_GB300_H */
