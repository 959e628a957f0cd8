// Batch pipeline: the next batch's host-to-device copy (and the previous
// pooled output's copy back) overlapped with the current step.
//
// Tencent PCG DataFun talk, "GPU 训练整体架构": every stage of the training
// step (reading, preprocessing, the GPU step) runs concurrently as a
// multi-stage pipeline; JD ads article 3.2.2: sparse updates pipelined with
// the next batch's data movement.  Here the stages on one GPU are: upload of
// batch t + 1 (copy stream), the step of batch t (the caller's compute
// stream: recording forward, then the recorded backward with the update),
// download of batch t - 1's pooled output (second copy stream).  The update
// of step t is ordered before the forward of step t + 1 on the compute
// stream, so results are exactly those of the same calls made one after the
// other; overlapping the update itself with the next forward would let that
// forward read rows half-updated (a stale, asynchronous update), which this
// pipeline does not do.
//
// Each in-flight batch owns one of `depth` buffer sets (CSR offsets and
// keys, optionally grad_out, the pooled output, the backward workspace).
// Batch t's upload into a set waits only for batch t - depth's backward (the
// last reader of the set's inputs), and batch t's forward, which writes the
// set's pooled output, waits for batch t - depth's download of it: the
// download of one batch never holds up the upload of a later one.  All
// waits are GPU-side (events), so the host never blocks except in
// emb_pipeline_wait.
#include <algorithm>
#include <vector>

#include "emb_internal.cuh"

namespace {

struct PipeSet {
  int64_t* offsets = nullptr;    // device int64[max_bags + 1]
  int64_t* keys = nullptr;       // device int64[max_nnz]
  float* grad = nullptr;         // device f32[max_batch * sum_dims] (only if grad is uploaded)
  float* out = nullptr;          // device f32[max_batch * sum_dims]
  void* ws = nullptr;            // backward workspace
  size_t ws_bytes = 0;
  cudaEvent_t uploaded = nullptr;   // the batch's CSR offsets and keys are on the device
  cudaEvent_t grad_up = nullptr;    // and its grad_out (uploaded after them: only the backward needs it)
  cudaEvent_t forwarded = nullptr;  // the forward wrote `out`
  cudaEvent_t bwd_done = nullptr;   // the backward (or, forward-only, the forward) finished
  cudaEvent_t downloaded = nullptr; // the download stream passed the batch's pooled-output copy
  cudaEvent_t released = nullptr;   // backward and download done (emb_pipeline_wait)
  long long ticket = -1;
  long long n_bags = 0, nnz = 0;
  int pool = 0;
  bool has_grad = false;
  enum { kFree, kSubmitted, kForwarded, kReleased } state = kFree;
};

}  // namespace

struct emb_pipeline {
  emb_table* table = nullptr;
  cudaStream_t compute = nullptr;  // caller's
  cudaStream_t up = nullptr, down = nullptr;
  long long max_bags = 0, max_nnz = 0;
  int depth = 0;
  bool grad_upload = false;
  long long next_ticket = 0;
  std::vector<PipeSet> sets;
};

namespace emb {

static void pipe_free(emb_pipeline* p) {
  if (!p) return;
  if (p->up) cudaStreamSynchronize(p->up);
  if (p->down) cudaStreamSynchronize(p->down);
  if (p->compute) cudaStreamSynchronize(p->compute);
  for (PipeSet& s : p->sets) {
    dfree(s.offsets);
    dfree(s.keys);
    dfree(s.grad);
    dfree(s.out);
    dfree(s.ws);
    if (s.uploaded) cudaEventDestroy(s.uploaded);
    if (s.grad_up) cudaEventDestroy(s.grad_up);
    if (s.forwarded) cudaEventDestroy(s.forwarded);
    if (s.bwd_done) cudaEventDestroy(s.bwd_done);
    if (s.downloaded) cudaEventDestroy(s.downloaded);
    if (s.released) cudaEventDestroy(s.released);
  }
  if (p->up) cudaStreamDestroy(p->up);
  if (p->down) cudaStreamDestroy(p->down);
  delete p;
}

static PipeSet* pipe_set(emb_pipeline* p, long long ticket) {
  if (ticket < 0) return nullptr;
  PipeSet& s = p->sets[(size_t)(ticket % p->depth)];
  return s.ticket == ticket ? &s : nullptr;
}

}  // namespace emb

using namespace emb;

extern "C" {

emb_status emb_pipeline_create(emb_table* table, int64_t max_bags, int64_t max_nnz, int depth, int upload_grad,
                               void* compute_stream, emb_pipeline** out) {
  if (!out) return fail(EMB_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!table || max_bags < 1 || max_nnz < 0 || depth < 2 || depth > 8)
    return fail(EMB_ERR_INVALID_ARG, "pipeline needs a table, max_bags >= 1, max_nnz >= 0 and depth in [2, 8]");
  if (max_bags % table->st.n_slots != 0) return fail(EMB_ERR_INVALID_ARG, "max_bags must be a multiple of n_slots");
  if (max_bags > EMB_MAX_BAGS || max_nnz > EMB_MAX_NNZ) return fail(EMB_ERR_UNSUPPORTED, "beyond EMB_MAX_* limits");
  emb_pipeline* p = new (std::nothrow) emb_pipeline();
  if (!p) return fail(EMB_ERR_OOM, "host allocation failed");
  p->table = table;
  p->compute = (cudaStream_t)compute_stream;
  p->max_bags = max_bags;
  p->max_nnz = max_nnz;
  p->depth = depth;
  p->grad_upload = upload_grad != 0;
  p->sets.resize((size_t)depth);
  auto body = [&]() -> emb_status {
    EMB_CUDA(cudaStreamCreateWithFlags(&p->up, cudaStreamNonBlocking));
    EMB_CUDA(cudaStreamCreateWithFlags(&p->down, cudaStreamNonBlocking));
    const size_t rows = (size_t)(max_bags / table->st.n_slots) * (size_t)table->st.sum_dims;
    size_t ws_bytes = 0;
    emb_status rc = emb_bwd_workspace_size(table, max_bags, max_nnz, &ws_bytes);
    if (rc != EMB_OK) return rc;
    for (PipeSet& s : p->sets) {
      EMB_CUDA(dmalloc((void**)&s.offsets, (size_t)(max_bags + 1) * 8));
      EMB_CUDA(dmalloc((void**)&s.keys, (size_t)std::max<int64_t>(max_nnz, 1) * 8));
      if (p->grad_upload) EMB_CUDA(dmalloc((void**)&s.grad, std::max<size_t>(rows, 1) * 4));
      EMB_CUDA(dmalloc((void**)&s.out, std::max<size_t>(rows, 1) * 4));
      EMB_CUDA(dmalloc(&s.ws, ws_bytes));
      s.ws_bytes = ws_bytes;
      EMB_CUDA(cudaEventCreateWithFlags(&s.uploaded, cudaEventDisableTiming));
      EMB_CUDA(cudaEventCreateWithFlags(&s.grad_up, cudaEventDisableTiming));
      EMB_CUDA(cudaEventCreateWithFlags(&s.forwarded, cudaEventDisableTiming));
      EMB_CUDA(cudaEventCreateWithFlags(&s.bwd_done, cudaEventDisableTiming));
      EMB_CUDA(cudaEventCreateWithFlags(&s.downloaded, cudaEventDisableTiming));
      EMB_CUDA(cudaEventCreateWithFlags(&s.released, cudaEventDisableTiming));
      // every set starts free
      EMB_CUDA(cudaEventRecord(s.bwd_done, p->up));
      EMB_CUDA(cudaEventRecord(s.downloaded, p->up));
      EMB_CUDA(cudaEventRecord(s.released, p->up));
    }
    return EMB_OK;
  };
  emb_status rc = body();
  if (rc != EMB_OK) {
    pipe_free(p);
    return rc;
  }
  *out = p;
  return EMB_OK;
}

emb_status emb_pipeline_destroy(emb_pipeline* pipe) {
  if (!pipe) return fail(EMB_ERR_INVALID_ARG, "pipeline is NULL");
  pipe_free(pipe);
  return EMB_OK;
}

emb_status emb_pipeline_submit(emb_pipeline* p, const int64_t* offsets_h, int64_t n_bags, const int64_t* keys_h,
                               int64_t nnz, const float* grad_out_h, int64_t* ticket_out) {
  if (!p || !ticket_out || !offsets_h || (nnz > 0 && !keys_h)) return fail(EMB_ERR_INVALID_ARG, "NULL argument");
  if (n_bags < 0 || nnz < 0 || n_bags > p->max_bags || nnz > p->max_nnz)
    return fail(EMB_ERR_INVALID_ARG, "batch larger than the pipeline's max_bags / max_nnz");
  if (n_bags % p->table->st.n_slots != 0) return fail(EMB_ERR_INVALID_ARG, "n_bags must be a multiple of n_slots");
  if (p->grad_upload != (grad_out_h != nullptr))
    return fail(EMB_ERR_INVALID_ARG, "grad_out_h must be given exactly when the pipeline uploads gradients");
  const long long t = p->next_ticket;
  PipeSet& s = p->sets[(size_t)(t % p->depth)];
  if (s.state == PipeSet::kSubmitted || s.state == PipeSet::kForwarded)
    return fail(EMB_ERR_INVALID_ARG, "the buffer set is still held by a batch whose backward (or release) has not been called");
  // the set's previous batch must have finished its backward (the last reader of the inputs)
  EMB_CUDA(cudaStreamWaitEvent(p->up, s.bwd_done, 0));
  EMB_CUDA(cudaMemcpyAsync(s.offsets, offsets_h, (size_t)(n_bags + 1) * 8, cudaMemcpyHostToDevice, p->up));
  if (nnz > 0) EMB_CUDA(cudaMemcpyAsync(s.keys, keys_h, (size_t)nnz * 8, cudaMemcpyHostToDevice, p->up));
  EMB_CUDA(cudaEventRecord(s.uploaded, p->up));
  // grad_out last: the forward can start as soon as the CSR batch is in
  if (grad_out_h) {
    const size_t bytes = (size_t)(n_bags / p->table->st.n_slots) * (size_t)p->table->st.sum_dims * 4;
    if (bytes) EMB_CUDA(cudaMemcpyAsync(s.grad, grad_out_h, bytes, cudaMemcpyHostToDevice, p->up));
  }
  EMB_CUDA(cudaEventRecord(s.grad_up, p->up));
  s.ticket = t;
  s.n_bags = n_bags;
  s.nnz = nnz;
  s.has_grad = grad_out_h != nullptr;
  s.state = PipeSet::kSubmitted;
  p->next_ticket = t + 1;
  *ticket_out = t;
  return EMB_OK;
}

emb_status emb_pipeline_forward(emb_pipeline* p, int64_t ticket, emb_pool pool, float* out_d, float* out_h,
                                float** out_used) {
  if (!p) return fail(EMB_ERR_INVALID_ARG, "pipeline is NULL");
  PipeSet* s = pipe_set(p, ticket);
  if (!s || s->state != PipeSet::kSubmitted) return fail(EMB_ERR_INVALID_ARG, "unknown ticket, or its forward already ran");
  float* out = out_d ? out_d : s->out;
  EMB_CUDA(cudaStreamWaitEvent(p->compute, s->uploaded, 0));
  // the set's previous batch's pooled output must have been copied out
  EMB_CUDA(cudaStreamWaitEvent(p->compute, s->downloaded, 0));
  emb_status rc = emb_lookup_fwd_record(p->table, s->offsets, s->n_bags, s->keys, s->nnz, pool, out, s->ws,
                                        s->ws_bytes, p->compute);
  if (rc != EMB_OK) return rc;
  EMB_CUDA(cudaEventRecord(s->forwarded, p->compute));
  if (out_h) {
    const size_t bytes = (size_t)(s->n_bags / p->table->st.n_slots) * (size_t)p->table->st.sum_dims * 4;
    EMB_CUDA(cudaStreamWaitEvent(p->down, s->forwarded, 0));
    if (bytes) EMB_CUDA(cudaMemcpyAsync(out_h, out, bytes, cudaMemcpyDeviceToHost, p->down));
    EMB_CUDA(cudaEventRecord(s->downloaded, p->down));
  }
  s->pool = (int)pool;
  s->state = PipeSet::kForwarded;
  if (out_used) *out_used = out;
  return EMB_OK;
}

// Hand a forwarded batch's set back: once the compute stream has passed this
// point and the download is done (the download stream records `released`).
static emb_status pipe_release(emb_pipeline* p, PipeSet* s) {
  EMB_CUDA(cudaEventRecord(s->bwd_done, p->compute));
  EMB_CUDA(cudaStreamWaitEvent(p->down, s->bwd_done, 0));
  EMB_CUDA(cudaEventRecord(s->released, p->down));
  s->state = PipeSet::kReleased;
  return EMB_OK;
}

// The backward of a forwarded batch with either optimizer; releases its set.
static emb_status pipe_backward(emb_pipeline* p, int64_t ticket, const float* grad_out_d, bool ftrl, float lr,
                                float eps, const emb_ftrl_params* fp) {
  if (!p) return fail(EMB_ERR_INVALID_ARG, "pipeline is NULL");
  PipeSet* s = pipe_set(p, ticket);
  if (!s || s->state != PipeSet::kForwarded) return fail(EMB_ERR_INVALID_ARG, "unknown ticket, or its forward has not run");
  const float* g = grad_out_d ? grad_out_d : (s->has_grad ? s->grad : nullptr);
  if (!g && s->n_bags > 0) return fail(EMB_ERR_INVALID_ARG, "no grad_out: pass one or upload it with the batch");
  if (!grad_out_d && s->has_grad) EMB_CUDA(cudaStreamWaitEvent(p->compute, s->grad_up, 0));
  emb_status rc = ftrl ? emb_bwd_ftrl_recorded(p->table, s->n_bags, s->nnz, (emb_pool)s->pool, g, fp, s->ws,
                                               s->ws_bytes, p->compute)
                       : emb_bwd_adagrad_recorded(p->table, s->n_bags, s->nnz, (emb_pool)s->pool, g, lr, eps, s->ws,
                                                  s->ws_bytes, p->compute);
  if (rc != EMB_OK) return rc;
  return pipe_release(p, s);
}

emb_status emb_pipeline_backward_adagrad(emb_pipeline* p, int64_t ticket, const float* grad_out_d, float lr,
                                         float eps) {
  return pipe_backward(p, ticket, grad_out_d, false, lr, eps, nullptr);
}

emb_status emb_pipeline_backward_ftrl(emb_pipeline* p, int64_t ticket, const float* grad_out_d,
                                      const emb_ftrl_params* params) {
  if (!params) return fail(EMB_ERR_INVALID_ARG, "FTRL parameters are NULL");
  return pipe_backward(p, ticket, grad_out_d, true, 0.f, 0.f, params);
}

emb_status emb_pipeline_release(emb_pipeline* p, int64_t ticket) {
  if (!p) return fail(EMB_ERR_INVALID_ARG, "pipeline is NULL");
  PipeSet* s = pipe_set(p, ticket);
  if (!s || s->state != PipeSet::kForwarded) return fail(EMB_ERR_INVALID_ARG, "unknown ticket, or not forwarded");
  return pipe_release(p, s);
}

emb_status emb_pipeline_wait(emb_pipeline* p, int64_t ticket) {
  if (!p || ticket < 0 || ticket >= p->next_ticket) return fail(EMB_ERR_INVALID_ARG, "bad pipeline or ticket");
  PipeSet* s = pipe_set(p, ticket);
  if (s) {
    if (s->state != PipeSet::kReleased) return fail(EMB_ERR_INVALID_ARG, "the ticket's backward (or release) has not been called");
    EMB_CUDA(cudaEventSynchronize(s->released));
  } else {
    // the set was handed to a later batch: this batch's release was recorded
    // on the download stream before anything that is there now
    EMB_CUDA(cudaStreamSynchronize(p->down));
  }
  return EMB_OK;
}

}  // extern "C"
