// fp64 row passes (int64 fixed-point butterflies).
#include "kernel_sets.cuh"

namespace fwt {
void register_rows_c64(std::vector<KernelEntry>& v) {
  RowSet<FWT_C64, 1, 1, double, ArithF64, 14>::add(v);
  v.push_back(cluster_entry<FWT_C64, 1, 13, 1>());  // 2^14-element vectors on CTA pairs
}
}  // namespace fwt
