// OSK with the GQA page union (osk_union_kernel.cuh): instances for head dimension 128.
#include "osk_union_kernel.cuh"

namespace cosa {

cudaError_t launch_osk_union_d128(const OskLaunch& L, cudaStream_t stream) {
  return launch_osk_union_hd<128>(L, stream);
}

}  // namespace cosa
