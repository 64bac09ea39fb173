// OSK instances for page size 16 (osk_kernel.cuh).
#include "osk_kernel.cuh"

namespace cosa {

cudaError_t launch_osk_p16(const OskLaunch& L, cudaStream_t stream) { return launch_osk_page<16>(L, stream); }

}  // namespace cosa
