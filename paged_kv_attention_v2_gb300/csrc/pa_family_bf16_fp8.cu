// pa_family_bf16_fp8.cu -- kernel instantiations for a bf16 query with an fp8
// (E4M3 or E5M2) KV cache.
#include "pa_launch.cuh"

namespace pa {
cudaError_t launch_bf16_fp8(const Params& p, const LaunchArgs& la, int kv) {
    return kv == kKvE4M3 ? launch_family<__nv_bfloat16, kKvE4M3>(p, la) : launch_family<__nv_bfloat16, kKvE5M2>(p, la);
}
}  // namespace pa
