// adamw_table_acc.cu -- AdamW with the grad read straight from the
// FlatParameter tensor table (adamw_table.cuh, ACC = true, PARTS = 1): the
// earlier micro-batches' fp32 sum is added first, g = fl(acc[k] +
// fl(grad_scale * x)); one table search per 2048-element part.
#include "adamw_table.cuh"

namespace zs {

ZS_DEBUG_UNIT(adamw_table_acc)

zero_status launch_adamw_table_acc(float* p, float* m, float* v, const float* acc, const zero_tensor* table,
                                   int n_tensors, int grad_dtype, int64_t shard_start, float gscale,
                                   const float* dscale, void* lowp, int lowp_dtype, int64_t n, const AdamScalars& s,
                                   const zero_adamw_device_state* ds, const zero_norm_result* clip, cudaStream_t st) {
  return launch_table_instance<true, 1>(p, m, v, acc, table, n_tensors, grad_dtype, shard_start, gscale, dscale,
                                        lowp, lowp_dtype, n, s, ds, clip, st);
}

}  // namespace zs
