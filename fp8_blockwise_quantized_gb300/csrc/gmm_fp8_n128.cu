// The single-CTA FP8 forward kernel's BN = 128 instances (plain output):
// 3, 4 (default) or 5 ring slots, 2 (default) or 4 TMEM partial buffers.
#include "gmm_fp8_kernel.cuh"

namespace gmm {

namespace {

template <int STAGES>
cudaError_t launch_stages(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                          const FwdArgs& args, int grid, cudaStream_t stream) {
  if (args.tmem_bufs == 4) return launch<128, false, false, STAGES, 4>(map_a, map_b, map_out, args, grid, stream);
  return launch<128, false, false, STAGES, 2>(map_a, map_b, map_out, args, grid, stream);
}

}  // namespace

cudaError_t launch_gmm_fp8_n128(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                                const FwdArgs& args, int grid, cudaStream_t stream) {
  if (args.stages == 3) return launch_stages<3>(map_a, map_b, map_out, args, grid, stream);
  if (args.stages == 5) return launch_stages<5>(map_a, map_b, map_out, args, grid, stream);
  return launch_stages<4>(map_a, map_b, map_out, args, grid, stream);
}

}  // namespace gmm
