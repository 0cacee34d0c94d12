// pa_family_f16.cu -- kernel instantiations for f16 storage (compiled on its own
// so the three storage types build in parallel).
#include "pa_launch.cuh"

namespace pa {
cudaError_t launch_f16(const Params& p, const LaunchArgs& la) { return launch_family<__half>(p, la); }
}  // namespace pa
