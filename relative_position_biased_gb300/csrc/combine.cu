// combine.cu -- log-sum-exp merge of split-KV partials (decode).
//
// Each split s of a row's key range produced a normalised partial output o_s
// and its logsumexp lse_s.  Softmax over the union of disjoint key sets gives
//     lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s,
// (the split-KV decode with num_splits on the page "vLLM Day-0 support for TML
// Inkling", paragraph on FA4 with sheared bias).
//
// RW warps share one (t, h) row: warp w takes splits w, w + RW, ...; each lane
// holds 4 of the 128 output columns.  The warps meet in shared memory for the
// max and for the final sums.  RW grows with the split count so long-context
// decode (hundreds of splits, few rows) keeps enough loads in flight.
#include "launch.h"

namespace relattn {
namespace {

constexpr int kCombineThreads = 256;

template <int RW>
__global__ void __launch_bounds__(kCombineThreads)
relattn_combine_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part,
                       int num_splits, int total_q, int num_heads, __nv_bfloat16 *__restrict__ out,
                       float *__restrict__ lse) {
  constexpr int kWarps = kCombineThreads / 32, kRowsPerCta = kWarps / RW;
  __shared__ float red_m[kWarps], red_z[kWarps];
  __shared__ float4 red_acc[kWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rsub = warp / RW, wi = warp % RW;
  // launched as a programmatic dependent of the split kernel: its partials
  // are complete and visible past this point (a plain launch returns at once)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long rows = (long)total_q * num_heads;
  const long row = (long)blockIdx.x * kRowsPerCta + rsub;
  const bool active = row < rows;

  float m = -INFINITY;
  if (active)
    for (int s = wi * 32 + lane; s < num_splits; s += RW * 32) m = fmaxf(m, lse_part[(long)s * rows + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (RW > 1) {
    if (lane == 0) red_m[warp] = m;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < RW; ++i) m = fmaxf(m, red_m[rsub * RW + i]);
  }

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float z = 0.f;
  if (active && m != -INFINITY) {
#pragma unroll 4
    for (int s = wi; s < num_splits; s += RW) {
      const float ls = lse_part[(long)s * rows + row];
      float4 v = *reinterpret_cast<const float4 *>(o_part + ((long)s * rows + row) * kHeadDim + lane * 4);
      // an empty split (lse = -inf) contributes nothing, whatever its o_s holds
      const bool empty = ls == -INFINITY;
      const float w = empty ? 0.f : exp2f((ls - m) * kLog2e);
      if (empty) v = make_float4(0.f, 0.f, 0.f, 0.f);
      z += w;
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
  }
  if (RW > 1) {
    red_acc[warp][lane] = acc;
    if (lane == 0) red_z[warp] = z;
    __syncthreads();
    if (wi != 0) return;
#pragma unroll
    for (int i = 1; i < RW; ++i) {
      const float4 o = red_acc[warp + i][lane];
      acc.x += o.x;
      acc.y += o.y;
      acc.z += o.z;
      acc.w += o.w;
      z += red_z[warp + i];
    }
  }
  if (!active) return;
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

template <int RW>
cudaError_t launch_rw(const float *o_part, const float *lse_part, int num_splits, int total_q,
                      int num_heads, __nv_bfloat16 *out, float *lse, cudaStream_t stream, bool pdl) {
  constexpr int kRowsPerCta = kCombineThreads / 32 / RW;
  const long rows = (long)total_q * num_heads;
  const unsigned blocks = (unsigned)((rows + kRowsPerCta - 1) / kRowsPerCta);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, relattn_combine_kernel<RW>, o_part, lse_part, num_splits, total_q,
                            num_heads, out, lse);
}

}  // namespace

cudaError_t launch_combine(const float *o_part, const float *lse_part, int num_splits, int total_q,
                           int num_heads, __nv_bfloat16 *out, float *lse, cudaStream_t stream, bool pdl) {
  const long rows = (long)total_q * num_heads;
  if (rows == 0) return cudaSuccess;
  if (num_splits >= 64) return launch_rw<8>(o_part, lse_part, num_splits, total_q, num_heads, out, lse, stream, pdl);
  if (num_splits >= 16) return launch_rw<4>(o_part, lse_part, num_splits, total_q, num_heads, out, lse, stream, pdl);
  if (num_splits >= 4) return launch_rw<2>(o_part, lse_part, num_splits, total_q, num_heads, out, lse, stream, pdl);
  return launch_rw<1>(o_part, lse_part, num_splits, total_q, num_heads, out, lse, stream, pdl);
}

}  // namespace relattn
