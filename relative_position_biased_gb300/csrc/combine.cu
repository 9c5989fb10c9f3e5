// combine.cu -- log-sum-exp merge of split-KV partials (decode).
//
// Each split s of a row's key range produced a normalised partial output o_s
// and its logsumexp lse_s.  Softmax over the union of disjoint key sets gives
//     lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s,
// which is what one warp per (t, h) row evaluates here (the split-KV decode
// with num_splits on the page "vLLM Day-0 support for TML Inkling", paragraph
// on FA4 with sheared bias).
#include "launch.h"

namespace relattn {
namespace {

constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32)
relattn_combine_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part,
                       int num_splits, int total_q, int num_heads, __nv_bfloat16 *__restrict__ out,
                       float *__restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const long rows = (long)total_q * num_heads;
  const long row = (long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  float m = -INFINITY;
  for (int s = 0; s < num_splits; ++s) m = fmaxf(m, lse_part[(long)s * rows + row]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float z = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < num_splits; ++s) {
      const float ls = lse_part[(long)s * rows + row];
      if (ls == -INFINITY) continue;
      const float w = exp2f((ls - m) * kLog2e);
      const float4 v = *reinterpret_cast<const float4 *>(o_part + ((long)s * rows + row) * kHeadDim + lane * 4);
      z += w;
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
  }
  const float inv = z > 0.f ? 1.f / z : 0.f;
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2 *>(out + row * kHeadDim + lane * 4) = packed;
  if (lane == 0) {
    const long t = row / num_heads, h = row - t * num_heads;
    lse[h * total_q + t] = z > 0.f ? m + logf(z) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_combine(const float *o_part, const float *lse_part, int num_splits, int total_q,
                           int num_heads, __nv_bfloat16 *out, float *lse, cudaStream_t stream) {
  const long rows = (long)total_q * num_heads;
  if (rows == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((rows + kCombineWarps - 1) / kCombineWarps);
  relattn_combine_kernel<<<blocks, kCombineWarps * 32, 0, stream>>>(o_part, lse_part, num_splits,
                                                                     total_q, num_heads, out, lse);
  return cudaGetLastError();
}

}  // namespace relattn
