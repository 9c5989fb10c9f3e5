// common.cuh -- shared device helpers and the internal launch descriptor for
// the relative-attention kernels (sm_103a).  Inline PTX wrappers are written
// from the PTX ISA's instruction descriptions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/relattn.h"

namespace relattn {

constexpr int kHeadDim = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device error word: kernels OR bits in, relattn_get_device_error reads it.
enum DeviceError : int {
  kDevErrSeqlens = 1,   // cu_seqlens inconsistent (Lk < Lq or above max_seqlen)
  kDevErrTimeout = 2,   // a bounded wait gave up
};

// A bounded wait at `site` gave up: set the timeout bit and, if no site is
// recorded yet, record this one in bits 8+ (the first CTA to report wins, so
// the word names one real wait site rather than an OR of several).
__device__ __forceinline__ void record_timeout(int *err, int site) {
  int old = *reinterpret_cast<volatile int *>(err);
  for (;;) {
    const int want = (old >> 8) ? (old | kDevErrTimeout) : (old | kDevErrTimeout | (site << 8));
    if (want == old) return;
    const int seen = atomicCAS(err, old, want);
    if (seen == old) return;
    old = seen;
  }
}

// Everything a kernel needs, resolved on the host from relattn_params.
struct KernelArgs {
  const __nv_bfloat16 *q, *k, *v, *r, *P;
  const int32_t *cu_q, *cu_k;
  __nv_bfloat16 *out;
  float *lse;
  float *o_part;     // decode split partials [S][total_q*Hq][128]
  float *lse_part;   // [S][total_q*Hq]
  int *err;          // device error word
  int batch, total_q, max_q, max_k, Hq, Hkv, group;
  int rd, rd_pad, E, window;
  float alpha_log2e;     // alpha * log2(e)
  float inv_ln_base;     // 1/ln(base), 0 when log-scale is off
  int num_splits, split_chunk;   // decode
  int q_tiles;                   // prefill: query tiles per (sequence, head)
  int row_blocks;                // decode: 128-row blocks per (sequence, kv head)
  int r_vec_ok, p_vec_ok;        // 16-byte vector loads allowed for r / P
  int test_skip_k_tile;          // test hook (tcgen05 kernels): never load this K tile; -1 = off
  int band_only;                 // prefill, bias kernel: only the key tiles of the bias band
  int init_from_out;             // prefill, main kernel: start from the band's out / lse
  int sms;                       // CTAs of a persistent launch: the SM count (or a test cap)
  // paged K / V (decode): keys at position p of sequence b sit at pool row
  // block_table[b * max_pages + p / page_size] * page_size + p % page_size;
  // block_table == nullptr: contiguous rows cu_seqlens_k[b] + p
  const int32_t *block_table;
  int page_size, max_pages, num_pages;
  // few-row decode (decode_tc.cu): R = r . P of every decode row and
  // distance < E, fp32 [total_q * Hq][E] in the workspace (null without a bias)
  const float *rdec;
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global->shared; when !pred the 16 bytes are zero-filled
// and nothing is read.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool pred) {
  const int n = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];\n"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Length-dependent log-scale s(i) = max(1, ln(i+1)/ln(base)) (1 when off).
__device__ __forceinline__ float log_scale(int pos, float inv_ln_base) {
  if (inv_ln_base <= 0.f) return 1.f;
  return fmaxf(1.f, logf(static_cast<float>(pos + 1)) * inv_ln_base);
}

}  // namespace relattn
