// Tensor-core (tcgen05 / TMEM / TMA) decode kernel -- placeholder until built.
#include "common.cuh"

namespace qkmla {
int launch_decode_tc(const qkmla_decode_args*, const DecodePlan&, cudaStream_t) { return QKMLA_ERR_UNSUPPORTED; }
}  // namespace qkmla
