// The single-CTA FP8 forward kernel's BN = 256 instances and the dispatch
// over all single-CTA instances (BN = 128 ones in gmm_fp8_n128.cu).
#include "gmm_fp8_kernel.cuh"

namespace gmm {

Fp8Geometry fp8_geometry(int N, int fuse, int bn) {
  if (fuse) return {256, 128, 128};
  if (bn == 256 || (bn == 0 && N % 256 == 0)) return {256, 256, 256};
  return {128, 128, 128};
}

namespace {

template <bool FUSE, bool QUANT>
cudaError_t launch_n256(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                        const FwdArgs& args, int grid, cudaStream_t stream) {
  if (args.stages == 2) return launch<256, FUSE, QUANT, 2, 2>(map_a, map_b, map_out, args, grid, stream);
  return launch<256, FUSE, QUANT, 3, 2>(map_a, map_b, map_out, args, grid, stream);
}

}  // namespace

cudaError_t launch_gmm_fp8(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                           const FwdArgs& args, int grid, cudaStream_t stream) {
  if (args.fuse && args.hq) return launch_n256<true, true>(map_a, map_b, map_out, args, grid, stream);
  if (args.fuse) return launch_n256<true, false>(map_a, map_b, map_out, args, grid, stream);
  if (args.bn == 256) return launch_n256<false, false>(map_a, map_b, map_out, args, grid, stream);
  return launch_gmm_fp8_n128(map_a, map_b, map_out, args, grid, stream);
}

}  // namespace gmm
