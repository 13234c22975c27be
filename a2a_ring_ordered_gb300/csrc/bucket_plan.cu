// bucket_plan.cu -- DDP gradient bucketing (host only).
//
// "dist_train", Communication-Computation Overlap: DDP cuts the gradients into
// buckets of at most bucket_cap_mb (25 MB by default) in the order backprop
// produces them and all-reduces a bucket as soon as every gradient in it is
// ready, overlapping that all-reduce with the rest of the backward pass.
//
// Rule: walk the gradients in the given (ready) order; a gradient joins the
// current bucket if the bucket's bytes stay within the cap, otherwise it
// starts a new bucket; a gradient larger than the cap gets a bucket of its
// own.  A bucket is the contiguous concatenation of its gradients.
#include "ccl_internal.h"

using ccl::report_error;

extern "C" ccl_status_t ccl_plan_buckets(const size_t* numel, size_t count, size_t elem_bytes,
                                         size_t cap_bytes, uint32_t* bucket_of, size_t* offset,
                                         size_t* bucket_numel, size_t* num_buckets) {
  ccl::clear_last_error();
  if (num_buckets == nullptr) return report_error(CCL_ERR_INVALID_ARG, "num_buckets is NULL");
  *num_buckets = 0;
  if (elem_bytes == 0 || cap_bytes < elem_bytes)
    return report_error(CCL_ERR_INVALID_ARG, "need elem_bytes > 0 and cap_bytes >= elem_bytes");
  if (count == 0) return CCL_OK;
  if (numel == nullptr || bucket_of == nullptr || offset == nullptr)
    return report_error(CCL_ERR_INVALID_ARG, "numel, bucket_of or offset is NULL");
  const size_t cap_elems = cap_bytes / elem_bytes;
  size_t b = 0, fill = 0, members = 0;  // current bucket, its elements and gradients
  for (size_t i = 0; i < count; ++i) {
    const size_t m = numel[i];
    // a bucket that already holds gradients is closed when this one would
    // take it past the cap
    if (members != 0 && (fill > cap_elems || m > cap_elems - fill)) {
      if (bucket_numel != nullptr) bucket_numel[b] = fill;
      ++b;
      fill = 0;
      members = 0;
    }
    ++members;
    if (b > 0xFFFFFFFEu) return report_error(CCL_ERR_INVALID_ARG, "more than 2^32-1 buckets");
    bucket_of[i] = static_cast<uint32_t>(b);
    offset[i] = fill;
    fill += m;
  }
  if (bucket_numel != nullptr) bucket_numel[b] = fill;
  *num_buckets = b + 1;
  return CCL_OK;
}
