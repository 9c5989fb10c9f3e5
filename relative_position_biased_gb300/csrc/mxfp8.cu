// mxfp8.cu -- MXFP8 quantisation of bf16 tensors (K / V caches, or any tensor
// whose rows are multiples of 32 elements).
//
// The page "SGLang and Miles Add Day-0 Support for Inkling", section
// "Relative Logits Optimization", paragraph "MXFP8 Support", stores K and V in
// MXFP8.  Format (OCP Microscaling): FP8 E4M3 elements, one E8M0 scale byte
// 2^(b - 127) per 32 consecutive elements.  A block's shared exponent is
// floor(log2(amax)) - 8 (8 = the exponent of E4M3's largest power of two),
// clamped to [-127, 127], -127 for an all-zero block; each element is
// x * 2^-e rounded to the nearest E4M3 value (ties to even, the sign kept,
// saturating at 448).
//
// One thread per 32-element block: 64 bytes in (four 16-byte loads), 32 code
// bytes and one scale byte out.  x * 2^-e is exact in fp32 wherever the
// result can round to a non-zero E4M3 value, so the codes are the exact
// round-to-nearest ones; the conversion itself is the hardware's
// round-to-nearest-even, saturating E4M3 conversion.
#include "launch.h"
#include "mxfp8.cuh"

namespace relattn {
namespace {

constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads)
relattn_quantize_mxfp8_kernel(const uint4 *__restrict__ x, long n_blocks, uint4 *__restrict__ codes,
                              uint8_t *__restrict__ scales) {
  const long blk = (long)blockIdx.x * kQuantThreads + threadIdx.x;
  if (blk >= n_blocks) return;
  uint32_t c[8];
  int e;
  quantize_block32(x + blk * 4, c, e);
  codes[blk * 2] = make_uint4(c[0], c[1], c[2], c[3]);
  codes[blk * 2 + 1] = make_uint4(c[4], c[5], c[6], c[7]);
  scales[blk] = (uint8_t)(e + 127);
}

}  // namespace

cudaError_t launch_quantize_mxfp8(const void *x, long n_blocks, void *codes, void *scales,
                                  cudaStream_t stream) {
  if (n_blocks <= 0) return cudaSuccess;
  const long grid = (n_blocks + kQuantThreads - 1) / kQuantThreads;
  if (grid > 0x7fffffffL) return cudaErrorInvalidValue;
  relattn_quantize_mxfp8_kernel<<<(unsigned)grid, kQuantThreads, 0, stream>>>(
      static_cast<const uint4 *>(x), n_blocks, static_cast<uint4 *>(codes), static_cast<uint8_t *>(scales));
  return cudaGetLastError();
}

}  // namespace relattn
