// OSK instances for page size 128 (osk_kernel.cuh).
#include "osk_kernel.cuh"

namespace cosa {

cudaError_t launch_osk_p128(const OskLaunch& L, cudaStream_t stream) { return launch_osk_page<128>(L, stream); }

}  // namespace cosa
