// Test probe: the largest relative error of the hardware base-2 exponential (ex2.approx.ftz.f32, the
// instruction the KAP block-score kernel takes exp with) over every fp32 input in a bit-pattern range,
// against the float64 exp2.  The KAP bounds |score - exact| with an assumed relative error of that
// instruction; a test compares the measured maximum with the assumption.  Test code only: built by
// the test that uses it, not part of libcosa.
//
//   ex2_error_probe(lo_bits, hi_bits, out, stream)
//     every float whose bit pattern lies in [lo_bits, hi_bits] (one sign; no NaN patterns) is an
//     input; out (device, 2 x uint64, zeroed by the caller) receives the bit patterns of the largest
//     relative error (a positive double, so its bits order like its value) and of its input.
//   Returns 0, or -3 for a CUDA launch error.
#include <cstdint>

#include <cuda_runtime.h>

#include "ptx.cuh"

namespace {

__global__ void ex2_probe_kernel(uint32_t lo, uint32_t hi, unsigned long long* out) {
  const uint64_t n = static_cast<uint64_t>(hi) - lo + 1;
  unsigned long long best = 0, arg = 0;
  for (uint64_t t = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
    const uint32_t bits = lo + static_cast<uint32_t>(t);
    const float x = __uint_as_float(bits);
    const double want = exp2(static_cast<double>(x));
    const double got = static_cast<double>(cosa::ex2_approx(x));
    const double rel = fabs(got - want) / want;
    const unsigned long long rb = static_cast<unsigned long long>(__double_as_longlong(rel));
    if (rb > best) {
      best = rb;
      arg = bits;
    }
  }
  // the largest error of the block, then one atomic per block
  __shared__ unsigned long long sb[256], sa[256];
  sb[threadIdx.x] = best;
  sa[threadIdx.x] = arg;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o && sb[threadIdx.x + o] > sb[threadIdx.x]) {
      sb[threadIdx.x] = sb[threadIdx.x + o];
      sa[threadIdx.x] = sa[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const unsigned long long prev = atomicMax(&out[0], sb[0]);
    if (sb[0] > prev) out[1] = sa[0];   // input of (one of) the largest errors; races only mislabel it
  }
}

}  // namespace

extern "C" int ex2_error_probe(uint32_t lo_bits, uint32_t hi_bits, void* out, void* stream) {
  if (hi_bits < lo_bits || out == nullptr) return -1;
  ex2_probe_kernel<<<4096, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      lo_bits, hi_bits, static_cast<unsigned long long*>(out));
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}
