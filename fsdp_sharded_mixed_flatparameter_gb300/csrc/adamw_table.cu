// adamw_table.cu -- AdamW with the grad read straight from the FlatParameter
// tensor table (adamw_table.cuh): the grad is fl(grad_scale * x) alone, one
// table search per 2048-element part; and the entry that picks the instance
// (the others: adamw_table_acc.cu, adamw_table_p4.cu, adamw_table_p4_acc.cu).
#include "adamw_table.cuh"

namespace zs {

ZS_DEBUG_UNIT(adamw_table)

zero_status launch_adamw_table(float* p, float* m, float* v, const float* acc, const zero_tensor* table,
                               int n_tensors, int grad_dtype, int64_t shard_start, float gscale, const float* dscale,
                               void* lowp, int lowp_dtype, int64_t n, const AdamScalars& s,
                               const zero_adamw_device_state* ds, const zero_norm_result* clip, cudaStream_t st) {
  const bool four = table_four_parts(n_tensors);
  AdamwTableInstance* const other = (acc != nullptr) ? (four ? launch_adamw_table_p4_acc : launch_adamw_table_acc)
                                    : (four ? launch_adamw_table_p4 : nullptr);
  if (other != nullptr)
    return other(p, m, v, acc, table, n_tensors, grad_dtype, shard_start, gscale, dscale, lowp, lowp_dtype, n, s, ds,
                 clip, st);
  return launch_table_instance<false, 1>(p, m, v, nullptr, table, n_tensors, grad_dtype, shard_start, gscale, dscale,
                                         lowp, lowp_dtype, n, s, ds, clip, st);
}

}  // namespace zs
