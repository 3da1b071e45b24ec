// kvq_decode_test_wait.cu -- the decode kernel instantiated with the wait
// limit carried in its parameters, launched only while a test has shortened
// that limit (kvq_test_set_wait_limit_ns) to exercise the timeout path
// without a hang; the kernel itself is in kvq_decode_kernel.cuh.
#include "kvq_decode_kernel.cuh"

namespace kvq {

kvq_status launch_decode_mma_test_wait(const DecodeParams& dp, cudaStream_t s, int ctas, bool after_append) {
  return dp.head_dim == 128 ? launch_decode<128, true>(dp, s, ctas, after_append)
                            : launch_decode<64, true>(dp, s, ctas, after_append);
}

}  // namespace kvq
