// OSK instances for page size 32 (osk_kernel.cuh).
#include "osk_kernel.cuh"

namespace cosa {

cudaError_t launch_osk_p32(const OskLaunch& L, cudaStream_t stream) { return launch_osk_page<32>(L, stream); }

}  // namespace cosa
