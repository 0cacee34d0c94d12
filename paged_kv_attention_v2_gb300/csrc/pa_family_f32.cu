// pa_family_f32.cu -- kernel instantiations for f32 storage (compiled on its own
// so the three storage types build in parallel).
#include "pa_launch.cuh"

namespace pa {
cudaError_t launch_f32(const Params& p, const LaunchArgs& la) { return launch_family<float>(p, la); }
}  // namespace pa
