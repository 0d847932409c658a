// Decode kernel instances for f16 KV pools.
#include "decode.cuh"

namespace far {
bool decode_config_f16(int D, int qvp, DecodeConfig* c) { return decode_config_kind<KV_F16>(D, qvp, c); }
int decode_occupancy_f16(int D, int qvp) { return decode_occupancy_kind<KV_F16>(D, qvp); }
cudaError_t decode_launch_f16(const DecodeParams& p, int D, int qvp, cudaStream_t st) {
  return decode_launch_kind<KV_F16>(p, D, qvp, st);
}
}  // namespace far
