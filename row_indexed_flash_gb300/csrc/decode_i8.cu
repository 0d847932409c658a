// Decode kernel instances for i8 KV pools.
#include "decode.cuh"

namespace far {
bool decode_config_i8(int D, int qvp, DecodeConfig* c) { return decode_config_kind<KV_I8>(D, qvp, c); }
int decode_occupancy_i8(int D, int qvp) { return decode_occupancy_kind<KV_I8>(D, qvp); }
cudaError_t decode_launch_i8(const DecodeParams& p, int D, int qvp, cudaStream_t st) {
  return decode_launch_kind<KV_I8>(p, D, qvp, st);
}
}  // namespace far
