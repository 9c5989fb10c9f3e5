// launch.h -- internal launchers called by the C ABI layer (api.cu).
#pragma once

#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace relattn {

// The calling thread's current CUDA context (a CUcontext, as an opaque key),
// or null before the runtime has made one current.  Per-device addresses the
// library caches (device symbols) are keyed on it: after cudaDeviceReset the
// primary context is new, the module is loaded again and the symbols may
// move, so a cached address is looked up again when the context changes.
inline void *current_cu_context() {
  static const PFN_cuCtxGetCurrent_v4000 get = []() -> PFN_cuCtxGetCurrent_v4000 {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    return nullptr;
  }();
  CUcontext c = nullptr;
  if (get && get(&c) != CUDA_SUCCESS) c = nullptr;
  return reinterpret_cast<void *>(c);
}

// Raise `func`'s dynamic shared-memory limit to `bytes` once per device.
// `done` holds one flag per device for that kernel; the first launch on a
// device sets the attribute under a process-wide lock, so host threads that
// launch concurrently neither race on the flag nor skip the call.
constexpr int kMaxDevicesAttr = 64;
inline cudaError_t set_max_smem_once(const void *func, int bytes,
                                     std::atomic<bool> (&done)[kMaxDevicesAttr]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesAttr)
    return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
  return e;
}

// Query rows per decode CTA for a given row count (max_seqlen_q * group).
int decode_warps_for_rows(int rows);

// Per-split key-chunk granularity (keys per tile) of the decode kernels.
constexpr int kDecodeKeyTile = 64;

size_t prefill_mma_smem_bytes(int rd_pad);
size_t decode_mma_smem_bytes(int warps, int rd_pad);

cudaError_t launch_prefill_mma(const KernelArgs &a, cudaStream_t stream);

// tcgen05 / TMA kernels: need 16-byte aligned q/k/v/out (and r/P), r_dim % 8 == 0,
// rel_extent % 8 == 0, r_dim <= 64 and at least one 128-key tile of K/V.
// Their key tiles (and decode split chunks) are kTcKeyTile keys.
constexpr int kTcKeyTile = 128;
bool tc_supported(const KernelArgs &a, int total_k);
cudaError_t launch_prefill_tc(const KernelArgs &a, int total_k, cudaStream_t stream);
// Prefill past the bias band (fwd_tc_main.cu): two query heads of one GQA
// group per CTA; needs an even group size, alpha > 0 and at least 128 query
// rows and keys.  With init_from_out it continues from the band kernel's
// out / lse (launched first with band_only).
bool tc_main_supported(const KernelArgs &a, int total_q, int total_k);
cudaError_t launch_prefill_tc_main(const KernelArgs &a, int total_k, cudaStream_t stream);
// decode on the same kernel: 128 rows of (token, head-in-group) per CTA; grid
// (num_splits, Hkv * row_blocks, batch); partials when num_splits > 1.
constexpr int kTcDecodeRows = 128;
cudaError_t launch_decode_tc(const KernelArgs &a, int total_k, cudaStream_t stream);
// decode of few rows (decode_tc.cu): keys along the MMA's M; an item is
// (split, sequence, kv head) and holds every row of the sequence's tokens for
// that kv head (max_q x group <= 16).  Needs 16-byte aligned q / k / v / out
// and at least 128 K / V rows.  With a bias it first computes R = r . P of the
// decode rows into a.rdec (decode_rel_bytes of workspace).  Partials when
// num_splits > 1.
constexpr int kFewRows = 16;
bool decode_few_rows_supported(const KernelArgs &a, int kv_rows);
size_t decode_rel_bytes(const KernelArgs &a);
cudaError_t launch_decode_few_rows(const KernelArgs &a, int kv_rows, cudaStream_t stream);
// The same decode on an MXFP8 K / V cache (decode_tc.cu): E4M3 codes k8 / v8
// [kv_rows, Hkv, 128] (16-byte aligned) with E8M0 scales ks / vs [kv_rows,
// Hkv, 4] (4-byte aligned); q quantised per item in the kernel, Q K^T as an
// E4M3 product per 32-dim block, V dequantised to bf16 for P V.  Contiguous
// K / V only.
bool decode_mxfp8_supported(const KernelArgs &a, const void *k8, const void *v8, const void *ks,
                            const void *vs, int kv_rows);
cudaError_t launch_decode_mxfp8(const KernelArgs &a, const void *k8, const void *v8, const void *ks,
                                const void *vs, int kv_rows, cudaStream_t stream);
// MXFP8 quantisation (mxfp8.cu): n_blocks blocks of 32 bf16 (x 16-byte
// aligned) -> 32 E4M3 codes (16-byte aligned) and one E8M0 scale byte each.
cudaError_t launch_quantize_mxfp8(const void *x, long n_blocks, void *codes, void *scales,
                                  cudaStream_t stream);
cudaError_t launch_decode_mma(const KernelArgs &a, int warps, cudaStream_t stream);
// pdl: launched as a programmatic dependent of the kernel before it on the
// stream (which lets it launch early; the combine waits for its results)
cudaError_t launch_combine(const float *o_part, const float *lse_part, int num_splits,
                           int total_q, int num_heads, __nv_bfloat16 *out, float *lse,
                           cudaStream_t stream, bool pdl = false);

// Backward pass (bwd_mma.cu): gradients of sum(dout * out) w.r.t. q, k, v, r.
struct BwdArgs {
  const __nv_bfloat16 *q, *k, *v, *r, *P, *out, *dout;
  const float *lse;            // [Hq, Tq] natural log (the forward's)
  const int32_t *cu_q, *cu_k;
  __nv_bfloat16 *dq, *dk, *dv, *dr;   // dr may be null (no bias)
  float *Dsum;                 // workspace [Hq, Tq]: dout . out
  float *Rall;                 // workspace [Tq, Hq, e_pad]: R = r . P for distances < E (bias only)
  int e_pad;                   // row stride of Rall: E rounded up to a multiple of 4
  int rall_ok;                 // 1: Rall has been written (the band's dq loads its R windows from it)
  float *dkv_part;             // workspace [2 halves][dk, dv][Tk, Hkv, 128] fp32 (GQA groups of 4, 6, 8 ...)
  int kv_split;                // 2: two tcgen05 dk / dv CTAs per key tile, each half the group's heads
  int test_skip_dkdv_step;     // test hooks: a step whose copies the tcgen05 dk / dv producer
  int test_skip_dq_step;       //   (or the tcgen05 dq producer) never issues (-1: off)
  float *dq_part;              // workspace [Tq, Hq, 128]: dq over the keys outside the bias band (fp32)
  int dq_split;                // 1: the tcgen05 dq takes the keys outside the band and writes
                               //    dq_part; the warp-MMA dq takes the band and adds dq_part
  int *err;
  int batch, total_q, total_k, max_q, max_k, Hq, Hkv, group;
  int rd, rd_pad, E, window;
  float alpha, alpha_log2e, inv_ln_base;
  int p_vec_ok;                // 16-byte vector loads of P allowed (E % 8 == 0)
  int q_tiles, k_tiles;        // 64-row / 64-key tiles per sequence (max)
};
size_t bwd_dq_smem_bytes(int rd_pad);
size_t bwd_dkdv_smem_bytes(int rd_pad);
cudaError_t launch_backward(const BwdArgs &a, int sms, cudaStream_t stream);
// dk / dv on tcgen05 (bwd_tc.cu): 16-byte aligned q / k / v / dout, r_dim <= 64,
// at least 128 keys and 64 query rows in total (the TMA boxes)
bool bwd_tc_supported(const BwdArgs &a);
cudaError_t launch_bwd_dkdv_tc(const BwdArgs &a, cudaStream_t stream);
// dq on tcgen05 (bwd_tc.cu) over the keys every row of a 128-row tile sees
// outside the bias band (all keys without a bias); also needs 128 query rows
bool bwd_dq_tc_supported(const BwdArgs &a);
cudaError_t launch_bwd_dq_tc(const BwdArgs &a, cudaStream_t stream);

// attention prologue (prologue.cu): ShortConv + Q/K RMSNorm + KV-cache rows;
// err = the device error word, sms = the SM count (sizes the grid),
// skip_tile = test hook (a token tile whose copies are never issued; -1 = off).
// mx: an MXFP8 cache to write as well (or instead, with null bf16 caches).
cudaError_t launch_prologue(const relattn_prologue_params *p, int *err, int sms, int skip_tile,
                            cudaStream_t stream, const relattn_kv_mxfp8_out *mx = nullptr);

}  // namespace relattn
