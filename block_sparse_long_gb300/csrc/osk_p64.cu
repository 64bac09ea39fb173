// OSK instances for page size 64 (osk_kernel.cuh).
#include "osk_kernel.cuh"

namespace cosa {

cudaError_t launch_osk_p64(const OskLaunch& L, cudaStream_t stream) { return launch_osk_page<64>(L, stream); }

}  // namespace cosa
