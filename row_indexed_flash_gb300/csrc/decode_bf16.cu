// Decode kernel instances for bf16 KV pools.
#include "decode.cuh"

namespace far {
bool decode_config_bf16(int D, int qvp, DecodeConfig* c) { return decode_config_kind<KV_BF16>(D, qvp, c); }
int decode_occupancy_bf16(int D, int qvp) { return decode_occupancy_kind<KV_BF16>(D, qvp); }
cudaError_t decode_launch_bf16(const DecodeParams& p, int D, int qvp, cudaStream_t st) {
  return decode_launch_kind<KV_BF16>(p, D, qvp, st);
}
}  // namespace far
