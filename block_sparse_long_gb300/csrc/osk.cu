// Ordered-Skipping Kernel (OSK): shared-memory sizes and the dispatch of a call to the instances
// of its page size (the kernel itself is in osk_kernel.cuh), or to the GQA page-union kernel
// (osk_union_kernel.cuh) under COSA_FLAG_GQA_UNION.
#include "osk_kernel.cuh"

namespace cosa {

size_t osk_smem_bytes(int block_size, int head_dim) {
  if (block_size == 128 && head_dim == 128) return sizeof(OskSmem<128, 128>) + 1024;
  if (block_size == 128 && head_dim == 64) return sizeof(OskSmem<128, 64>) + 1024;
  if (block_size == 64 && head_dim == 128) return sizeof(OskSmem<64, 128>) + 1024;
  return sizeof(OskSmem<64, 64>) + 1024;
}

cudaError_t launch_osk_union_d64(const OskLaunch& L, cudaStream_t stream);
cudaError_t launch_osk_union_d128(const OskLaunch& L, cudaStream_t stream);

cudaError_t launch_osk(const OskLaunch& L, cudaStream_t stream) {
  if (L.flags & COSA_FLAG_GQA_UNION) {
    if (L.block_size != 128) return cudaErrorInvalidValue;
    return L.head_dim == 128 ? launch_osk_union_d128(L, stream) : launch_osk_union_d64(L, stream);
  }
  switch (L.page_size) {
    case 16: return launch_osk_p16(L, stream);
    case 32: return launch_osk_p32(L, stream);
    case 64: return launch_osk_p64(L, stream);
    case 128: return launch_osk_p128(L, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cosa
