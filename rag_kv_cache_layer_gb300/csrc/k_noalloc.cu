// Deviation ranking for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc: code that enqueues work while
// another component owns every device allocation (an inference engine's
// memory pool, a plugin host), or that runs where an allocation's implicit
// device synchronisation is not acceptable.  For them
// cb_kv_deviation_topk_noalloc keeps the per-token deviations -- the
// scratch that cb_kv_deviation_topk takes from the caller -- in a
// file-scope device array of fixed size instead.  The caller still passes
// its inputs and the selected-index output.
//
// The array holds kNoAllocMaxCtx floats (4 MiB) on every device that loads
// the library, until the process exits.  All calls share it and it keeps
// the last call's contents; each call first writes every deviation it later
// reads, so nothing has to start at zero.  Calls whose execution overlaps on
// the GPU (concurrent streams, other threads) race on the array and must be
// serialised by the caller.
#include <mutex>
#include <vector>

#include "cb_common.cuh"
#include "cb_internal.h"

namespace cb {

constexpr int64_t kNoAllocMaxCtx = 1 << 20;   // context tokens per call

static __device__ __align__(256) float g_noalloc_dev[kNoAllocMaxCtx];

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is resolved
// once per device (with that device current) and cached.
static cudaError_t noalloc_scratch(float **out) {
  static std::mutex mu;
  static float *ptrs[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    float *p = nullptr;
    e = cudaGetSymbolAddress((void **)&p, g_noalloc_dev);
    if (e != cudaSuccess) return e;
    ptrs[dev] = p;
  }
  *out = ptrs[dev];
  return cudaSuccess;
}

}  // namespace cb

using namespace cb;

extern "C" cb_status cb_kv_deviation_topk_noalloc(const void *k_fresh, int64_t ld_fresh,
                                                  const void *k_reused, int64_t ld_reused,
                                                  int row_elems, cb_dtype dtype,
                                                  const cb_select_req *reqs, int n_req,
                                                  cb_policy policy, int32_t *idx_out,
                                                  cb_stream stream) {
  if (!k_fresh || !k_reused || !idx_out) return record_error(CB_ERR_INVALID_ARG, "NULL pointer");
  if (dtype != CB_F32 && dtype != CB_BF16) return record_error(CB_ERR_INVALID_ARG, "bad dtype");
  const size_t eb = dtype == CB_BF16 ? 2 : 4;
  if (row_elems <= 0 || (row_elems * eb) % 16 || ld_fresh < row_elems || ld_reused < row_elems ||
      (ld_fresh * eb) % 16 || (ld_reused * eb) % 16 || ((uintptr_t)k_fresh & 15) ||
      ((uintptr_t)k_reused & 15))
    return record_error(CB_ERR_INVALID_ARG, "rows must be 16-byte aligned and ld >= row_elems");
  if (n_req < 0 || n_req > CB_MAX_BATCH) return record_error(CB_ERR_INVALID_ARG, "n_req must be in [0, CB_MAX_BATCH]");
  if (n_req > 0 && !reqs) return record_error(CB_ERR_INVALID_ARG, "reqs is NULL");
  // dev_offset is not an input of this entry point (the deviations are
  // packed below), so whatever the caller left in it is not validated
  std::vector<cb_select_req> rq(reqs, reqs + n_req);
  for (cb_select_req &r : rq) r.dev_offset = 0;
  SelPlan plan;
  const char *err = "";
  if (make_sel_plan(rq.data(), n_req, policy, plan, &err) != CB_OK)
    return record_error(CB_ERR_INVALID_ARG, err);
  // deviations are packed request after request into the static array
  int64_t total = 0;
  for (SelReq &r : plan.reqs) {
    r.dev_offset = (int)total;
    total += r.n_ctx;
    if (total > kNoAllocMaxCtx)
      return record_error(CB_ERR_INVALID_ARG,
                          "cb_kv_deviation_topk_noalloc: more than 1048576 context tokens in one "
                          "call (the fixed scratch limit); split the call");
  }
  float *dev = nullptr;
  cudaError_t e = noalloc_scratch(&dev);
  if (e != cudaSuccess) return record_error(CB_ERR_CUDA, cudaGetErrorString(e));
  int *st = device_status_ptr();
  if (!st) return record_error(CB_ERR_CUDA, "cannot resolve the device status word");
  e = launch_deviation(k_fresh, ld_fresh, k_reused, ld_reused, row_elems, dtype,
                       plan.reqs.data(), (int)plan.reqs.size(), dev, stream);
  if (e == cudaSuccess) e = launch_selection(dev, plan, idx_out, st, stream);
  if (e != cudaSuccess) return record_error(CB_ERR_CUDA, cudaGetErrorString(e));
  return CB_OK;
}
