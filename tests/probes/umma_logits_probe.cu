// Test probe: every fp32 logit q . k of bf16 query and key rows, computed by the tensor cores in the
// operand layout of the KAP logits kernel: 128 x d tiles loaded by TMA with the 128-byte swizzle
// ([d / 64][128 rows][128 B], K-major), one tcgen05.mma of kind::f16 (bf16 in, fp32 accumulate) per
// 16-wide step of d into a 128 x 128 TMEM accumulator, read back with tcgen05.ld.
//
// The KAP certifies its selections with the bound |fp32 logit - exact| <= kappa * ||q|| * ||k||
// (CoSA Sec. 4.2, Eqs. (9)-(13) rank on these logits); this probe lets a test measure the tensor
// cores' accumulation error on adversarial inputs against that bound.  Test code only: it is built
// by the test that uses it and is not part of libcosa.
//
//   umma_logits_probe(q, k, out, rows_q, rows_k, d, status, stream)
//     q    bf16 [rows_q, d], k bf16 [rows_k, d] (device, 16-byte aligned), rows multiples of 128,
//     out  fp32 [rows_q, rows_k] (device), d in {64, 128};
//     status: device int32 the caller zeroes; a bounded wait that runs out writes -4 there.
//   Returns 0, -1 for bad arguments, -3 for a CUDA error.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "ptx.cuh"

namespace {

using namespace cosa;

template <int HD>
struct alignas(1024) ProbeSmem {
  uint8_t q[128 * HD * 2];
  uint8_t k[128 * HD * 2];
  uint64_t full, done;
  uint32_t tmem_base;
  int32_t abort_flag;
};

// 128 threads: warp 0 issues the TMA loads, warp 1 owns TMEM and issues the products, and all four
// warps read the accumulator (warp w reads TMEM lanes 32 w .. 32 w + 31).
template <int HD>
__global__ void __launch_bounds__(128) probe_kernel(const __grid_constant__ CUtensorMap qmap,
                                                    const __grid_constant__ CUtensorMap kmap, float* out,
                                                    int rows_k, int* status) {
  using S = ProbeSmem<HD>;
  constexpr int DH = HD / 64;
  extern __shared__ uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * 128, col0 = blockIdx.y * 128;
  if (threadIdx.x == 0) {
    mbar_init(&sm.full, 1);
    mbar_init(&sm.done, 1);
    sm.abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;
  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(&sm.full, 2 * 128 * HD * 2);
    for (int dh = 0; dh < DH; ++dh) {
      tma_load_2d(&sm.q[dh * 128 * 128], &qmap, &sm.full, dh * 64, row0);
      tma_load_2d(&sm.k[dh * 128 * 128], &kmap, &sm.full, dh * 64, col0);
    }
  }
  if (warp == 1 && lane == 0) {
    if (wait_parity_bounded(&sm.full, 0, abort_flag, status)) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint64_t ad = smem_desc_sw128(smem_u32(&sm.q[(kk >> 2) * 128 * 128 + (kk & 3) * 32]), 16, 1024);
        const uint64_t bd = smem_desc_sw128(smem_u32(&sm.k[(kk >> 2) * 128 * 128 + (kk & 3) * 32]), 16, 1024);
        umma_ss(tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
    }
    umma_commit(&sm.done);   // also when nothing was issued: the readers then stop on the abort flag
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, wait_parity_bounded(&sm.done, 0, abort_flag, status)) && !*abort_flag;
  if (ok) {
    tc_fence_after();
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    float* orow = out + static_cast<size_t>(row0 + warp * 32 + lane) * rows_k + col0;
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_addr + c, r);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4*>(orow + c + e) = make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                                                                __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
    }
  }
  // the loads landed before the products were issued; if they were not issued, wait for the loads
  if (warp == 0 && lane == 0 && *abort_flag) wait_parity_bounded(&sm.full, 0, nullptr, nullptr);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool encode(CUtensorMap* map, const void* base, int rows, int d) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t es[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HD>
int launch(const void* q, const void* k, float* out, int rows_q, int rows_k, int* status, cudaStream_t stream) {
  CUtensorMap qmap, kmap;
  if (!encode(&qmap, q, rows_q, HD) || !encode(&kmap, k, rows_k, HD)) return -3;
  const size_t smem = sizeof(ProbeSmem<HD>) + 1024;
  if (cudaFuncSetAttribute(probe_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return -3;
  probe_kernel<HD><<<dim3(rows_q / 128, rows_k / 128), 128, smem, stream>>>(qmap, kmap, out, rows_k, status);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace

extern "C" int umma_logits_probe(const void* q, const void* k, float* out, int rows_q, int rows_k, int d, int* status,
                                 void* stream) {
  if (q == nullptr || k == nullptr || out == nullptr || status == nullptr) return -1;
  if (rows_q < 128 || rows_k < 128 || rows_q % 128 != 0 || rows_k % 128 != 0) return -1;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(out)) % 16 != 0)
    return -1;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 128) return launch<128>(q, k, out, rows_q, rows_k, status, s);
  if (d == 64) return launch<64>(q, k, out, rows_q, rows_k, status, s);
  return -1;
}
