// OSK with the GQA page union (osk_union_kernel.cuh): instances for head dimension 64.
#include "osk_union_kernel.cuh"

namespace cosa {

cudaError_t launch_osk_union_d64(const OskLaunch& L, cudaStream_t stream) {
  return launch_osk_union_hd<64>(L, stream);
}

}  // namespace cosa
