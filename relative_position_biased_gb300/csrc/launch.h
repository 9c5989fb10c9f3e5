// launch.h -- internal launchers called by the C ABI layer (api.cu).
#pragma once

#include "common.cuh"

namespace relattn {

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
cudaError_t launch_decode_mma(const KernelArgs &a, int warps, cudaStream_t stream);
cudaError_t launch_combine(const float *o_part, const float *lse_part, int num_splits,
                           int total_q, int num_heads, __nv_bfloat16 *out, float *lse,
                           cudaStream_t stream);

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
  int test_skip_step;          // test hook: a step whose copies the tcgen05 producers never issue (-1 off)
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
cudaError_t launch_prologue(const relattn_prologue_params *p, int *err, int sms, int skip_tile,
                            cudaStream_t stream);

}  // namespace relattn
