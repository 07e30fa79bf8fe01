// int4 weight preparation (moe_repack_int4): the packed order of the codes,
// two per byte with the low nibble holding the even K index, becomes the
// paired order the converters of the int4 GEMM read with three shifts and four
// logic operations per 8 codes: within every 4-byte word (K indices k0..k7 of
// one row) the nibbles of the low 16 bits hold k0, k2, k4, k6 and those of the
// high 16 bits k1, k3, k5, k7, lowest first.  A pure permutation of nibbles,
// in place or out of place, bandwidth-bound.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kRepackThreads = 256;

__device__ __forceinline__ uint32_t pair_codes(uint32_t w) {
  uint32_t r = 0;
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    const uint32_t code = (w >> (4 * n)) & 0xFu;
    const int pos = (n & 1) ? 4 + (n >> 1) : (n >> 1);  // even K: nibble n/2, odd: 4 + n/2
    r |= code << (4 * pos);
  }
  return r;
}

// 16-byte vectors [0, n_vec), then single words [4 n_vec, n_words).
__global__ void __launch_bounds__(kRepackThreads)
    repack_int4_kernel(const uint32_t* in, uint32_t* out, size_t n_vec, size_t n_words) {
  pdl_wait();
  pdl_trigger();
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  const size_t i0 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const uint4* in4 = reinterpret_cast<const uint4*>(in);
  uint4* out4 = reinterpret_cast<uint4*>(out);
  for (size_t i = i0; i < n_vec; i += stride) {
    uint4 v = in4[i];
    v.x = pair_codes(v.x);
    v.y = pair_codes(v.y);
    v.z = pair_codes(v.z);
    v.w = pair_codes(v.w);
    out4[i] = v;
  }
  for (size_t i = 4 * n_vec + i0; i < n_words; i += stride) out[i] = pair_codes(in[i]);
}

}  // namespace

cudaError_t launch_repack_int4(const uint32_t* in, uint32_t* out, size_t n_words, cudaStream_t s) {
  if (n_words == 0) return cudaSuccess;
  const bool vec = (reinterpret_cast<uintptr_t>(in) % 16 == 0) && (reinterpret_cast<uintptr_t>(out) % 16 == 0);
  const size_t n_vec = vec ? n_words / 4 : 0;
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const size_t work = n_vec > 0 ? n_vec : n_words;
  size_t blocks = (work + kRepackThreads - 1) / kRepackThreads;
  const size_t cap = static_cast<size_t>(sms) * 8;  // grid-stride beyond 8 blocks per SM
  if (blocks > cap) blocks = cap;
  return launch_pdl(repack_int4_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kRepackThreads), 0, s, in, out,
                    n_vec, n_words);
}

}  // namespace moe
