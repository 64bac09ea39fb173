// Ordered-Skipping Kernel (OSK): shared-memory sizes and the dispatch of a call to the instances
// of its page size (the kernel itself is in osk_kernel.cuh).
#include "osk_kernel.cuh"

namespace cosa {

size_t osk_smem_bytes(int block_size, int head_dim) {
  if (block_size == 128 && head_dim == 128) return sizeof(OskSmem<128, 128>) + 1024;
  if (block_size == 128 && head_dim == 64) return sizeof(OskSmem<128, 64>) + 1024;
  if (block_size == 64 && head_dim == 128) return sizeof(OskSmem<64, 128>) + 1024;
  return sizeof(OskSmem<64, 64>) + 1024;
}

cudaError_t launch_osk(const OskLaunch& L, cudaStream_t stream) {
  switch (L.page_size) {
    case 16: return launch_osk_p16(L, stream);
    case 32: return launch_osk_p32(L, stream);
    case 64: return launch_osk_p64(L, stream);
    case 128: return launch_osk_p128(L, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cosa
