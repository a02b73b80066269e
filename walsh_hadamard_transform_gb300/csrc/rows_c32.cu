// fp32 row passes.
#include "kernel_sets.cuh"

namespace fwt {
void register_rows_c32(std::vector<KernelEntry>& v) {
  RowSet<FWT_C32, 0, 2, float, ArithF32, 15>::add(v);
  PhaseSet::add(v);
  ClusterSet<FWT_C32, 0>::add(v);
}
}  // namespace fwt
