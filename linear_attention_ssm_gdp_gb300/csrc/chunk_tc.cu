// Tensor-core (tcgen05) chunked forward: not built yet; every problem goes
// through the generic path.
#include "gdp_internal.cuh"

namespace gdp {

bool tc_supported(int, int, int, int, int, int, gdp_dtype) { return false; }

WsLayout tc_layout(int B, int T, int N_seq, int H, int HV, int K, int V, int M, int BT) {
  return generic_layout(B, T, N_seq, H, HV, K, V, M, BT);
}

cudaError_t launch_chunk_tc(const ChunkProblem&, const WsLayout&, uint8_t*) {
  return cudaErrorNotSupported;
}

}  // namespace gdp
