// Instantiations of the format-parameterised tensor-core decode kernel (tq_decode_mma.cuh) at
// head_dim 64: every pair of K code width (q8_0 = 0, turbo2/3/4 = 2/3/4) and V code width
// (q8_0 = 0, turbo2/3/4_mse = 1/2/3).
#include "tq_decode_mma.cuh"

namespace tq {

bool mma_has_d64(int wk, int wv) {
  if (wk != 0 && (wk < 2 || wk > 4)) return false;
  if (wv < 0 || wv > 3) return false;

  return true;
}

cudaError_t mma_launch_d64(const DecodeLaunch& k, int wk, int wv, int sm_count, cudaStream_t s) {
  using namespace mmad;
#define TQ_MMA_CASE(WK, WV) \
  case WK * 4 + WV:         \
    return launch_mma<Fmt<64, WK, WV>>(k, sm_count, s);
  if (!mma_has_d64(wk, wv)) return cudaErrorInvalidValue;
  switch (wk * 4 + wv) {
    TQ_MMA_CASE(0, 0) TQ_MMA_CASE(0, 1) TQ_MMA_CASE(0, 2) TQ_MMA_CASE(0, 3)
    TQ_MMA_CASE(2, 0) TQ_MMA_CASE(2, 1) TQ_MMA_CASE(2, 2) TQ_MMA_CASE(2, 3)
    TQ_MMA_CASE(3, 0) TQ_MMA_CASE(3, 1) TQ_MMA_CASE(3, 2) TQ_MMA_CASE(3, 3)
    TQ_MMA_CASE(4, 0) TQ_MMA_CASE(4, 1) TQ_MMA_CASE(4, 2) TQ_MMA_CASE(4, 3)
  }
#undef TQ_MMA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace tq
