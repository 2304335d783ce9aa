// engine_tc.cu -- split-K engine with tcgen05 tensor-core tiles (not built yet).
#include "engine.cuh"

namespace ssd {

size_t engine_tc_smem_bytes(int) { return 0; }

cudaError_t launch_engine_tc(int, const CUtensorMap &, const CUtensorMap &,
                             const EngineParams &, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace ssd
