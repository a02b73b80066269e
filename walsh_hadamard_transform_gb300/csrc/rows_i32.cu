// int32 row passes (wrapping add/sub).
#include "kernel_sets.cuh"

namespace fwt {
void register_rows_i32(std::vector<KernelEntry>& v) {
  RowSet<FWT_I32, 2, 2, uint32_t, ArithU32, 15>::add(v);
  ClusterSet<FWT_I32, 2>::add(v);
}
}  // namespace fwt
