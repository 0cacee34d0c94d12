// pa_family_bf16.cu -- kernel instantiations for bf16 storage (compiled on its own
// so the three storage types build in parallel).
#include "pa_launch.cuh"

namespace pa {
cudaError_t launch_bf16(const Params& p, const LaunchArgs& la) { return launch_family<__nv_bfloat16>(p, la); }
}  // namespace pa
