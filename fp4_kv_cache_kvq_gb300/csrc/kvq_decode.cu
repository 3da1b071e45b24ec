// kvq_decode.cu -- the decode kernel's production instantiations (the fixed
// ~2 s limit on its waits); the kernel itself is in kvq_decode_kernel.cuh.
#include "kvq_decode_kernel.cuh"

namespace kvq {

kvq_status launch_decode_mma(const DecodeParams& dp, cudaStream_t s, int ctas, bool after_append) {
  return dp.head_dim == 128 ? launch_decode<128, false>(dp, s, ctas, after_append)
                            : launch_decode<64, false>(dp, s, ctas, after_append);
}

}  // namespace kvq
