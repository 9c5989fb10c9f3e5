// bwd_tc.cu -- dk / dv of the relative-attention backward on tcgen05 / TMEM /
// TMA (key-major), P frozen.
//
// What a CTA computes (page "SGLang and Miles Add Day-0 Support for Inkling",
// section "Customized Efficient Kernels for Train-Inference Consistency",
// paragraph "Relative attention"; the chain rule through the softmax): for
// 128 keys j of one kv head and every (query head of the group, 64-row query
// tile) that sees them,
//     S^T = K Q^T,  dP^T = V dout^T                       (tcgen05, M = 128 keys, N = 64)
//     P^T = exp(s_i (alpha S^T + bias) - lse_i),  dS^T = s_i alpha P^T (dP^T - D_i)
//     dV += P^T dout,  dK += dS^T Q                        (tcgen05, A = P^T / dS^T in TMEM)
// with bias(i, j) = [0 <= i-j < E] R[i][i-j], R = r . P.
//
// Roles (12 warps): warp 0 the TMA producer (K / V once, q / dout per step);
// warp 1 the MMA issuer; warp 2 the per-step query constants (lse, D,
// log-scale) and, for steps inside the bias band, a TMA load of the R
// window R[i][cb + c] = r_i . P[:, cb + c] from the R array a pre-pass wrote;
// warps 4-11 two per key row (half the query columns each): they read S^T /
// dP^T rows from TMEM,
// gather the bias from the R window (lanes are consecutive keys, so every
// gather is one conflict-free row of the window), and write P^T / dS^T back
// into TMEM as bf16 for the dV / dK MMAs.  At the end they read dK / dV out.
//
// TMEM (512 columns): dK [0,128), dV [128,256), S^T buffers [256,320) and
// [320,384), dP^T buffers [384,448) and [448,512); P^T / dS^T (bf16 pairs)
// over columns [0,16) and [32,48) of their buffers: each elementwise warp
// packs its 32 query columns over the first half of the 32 it has read.
// S^T / dP^T of step n+1 are computed while the elementwise warps work on
// step n.
//
// Every wait is bounded; a timeout sets the device error word, the roles stop,
// the producer and the MMA issuer drain their own operations, TMEM is freed.
#include <cudaTypedefs.h>

#include <algorithm>

#include "launch.h"
#include "tc_common.cuh"

namespace relattn {
namespace {

using namespace tc;

constexpr int KT = 128;          // keys per CTA (MMA M)
constexpr int QT = 64;           // query rows per step (MMA N of S^T, K of dV / dK)
constexpr int QSTAGES = 3;
constexpr int NTHR = 384;         // 4 role warps + 8 elementwise warps
constexpr int NELEM = 256;        // elementwise threads (two per key row)
constexpr int RWC = 200;         // R window columns (distances cb .. cb + 199), one TMA box
constexpr int RWS = 200;         // fp32 row stride of the R window

// TMEM columns
constexpr uint32_t TM_DK = 0, TM_DV = 128, TM_ST = 256, TM_DP = 384;

// shared memory (offsets from a 1024-aligned base)
constexpr uint32_t SM_K = 0;                          // 2 boxes [128 keys x 128 B]
constexpr uint32_t SM_V = SM_K + 32768;
constexpr uint32_t SM_Q = SM_V + 32768;               // QSTAGES x 2 boxes [64 rows x 128 B]
constexpr uint32_t SM_DO = SM_Q + QSTAGES * 16384;
constexpr uint32_t SM_RW = SM_DO + QSTAGES * 16384;   // R window [64][RWS] fp32 (TMA box)
constexpr uint32_t SM_AUX = SM_RW + QT * RWS * 4;     // QSTAGES x {lse2, D, s*log2e, s*alpha} [64] fp32
constexpr uint32_t SM_BAR = SM_AUX + QSTAGES * 4 * QT * 4;
enum {
  B_KV_FULL = 0,
  B_Q_FULL = 1,                  // + stage
  B_Q_EMPTY = B_Q_FULL + QSTAGES,
  B_AUX_FULL = B_Q_EMPTY + QSTAGES,
  B_AUX_EMPTY = B_AUX_FULL + QSTAGES,
  B_S_FULL = B_AUX_EMPTY + QSTAGES,   // + buffer
  B_P_FULL = B_S_FULL + 2,            // + buffer
  B_R_FULL = B_P_FULL + 2,            // R window of a band step landed (TMA)
  B_RW_READ = B_R_FULL + 1,           // ... gathered (elementwise, all warps)
  B_DONE = B_RW_READ + 1,
  B_DRAIN = B_DONE + 1,
  B_COUNT = B_DRAIN + 1
};
constexpr uint32_t SM_TMEM_SLOT = SM_BAR + B_COUNT * 8;
constexpr uint32_t SM_ABORT = SM_TMEM_SLOT + 8;
constexpr uint32_t SM_TOTAL = SM_ABORT + 8;
constexpr uint32_t SMEM_BYTES_BWD = SM_TOTAL + 1024;
static_assert(SMEM_BYTES_BWD <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ int floor8(int x) { return x & ~7; }

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_test_wait(bar, parity))
    if (clock64() - t0 > 200000000ll) return false;
  return true;
}

__global__ void __launch_bounds__(NTHR, 1)
relattn_bwd_dkdv_tc_kernel(const __grid_constant__ BwdArgs a,
                           const __grid_constant__ CUtensorMap map_k,
                           const __grid_constant__ CUtensorMap map_v,
                           const __grid_constant__ CUtensorMap map_q,
                           const __grid_constant__ CUtensorMap map_do,
                           const __grid_constant__ CUtensorMap map_r) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sb = smem_addr(smem);
  auto bar = [&](int i) { return sb + SM_BAR + 8u * i; };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM_ABORT);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ------------------------------------------------------------ the CTA's keys and steps
  // blockIdx.y = kv head x kv_split: with a split, CTA half `half` takes
  // query heads [half * hpc, half * hpc + hpc) of the group
  const int g = blockIdx.y / a.kv_split, half = blockIdx.y - g * a.kv_split, b = blockIdx.z;
  const int hpc = a.group / a.kv_split;
  const int cq = a.cu_q[b], ck = a.cu_k[b];
  const int Lq = a.cu_q[b + 1] - cq, Lk = a.cu_k[b + 1] - ck;
  if (Lq < 0 || Lk < Lq || Lq > a.max_q || Lk > a.max_k) {
    if (tid == 0) atomicOr(a.err, kDevErrSeqlens);
    return;
  }
  const int j0 = blockIdx.x * KT;
  const int nkeys = min(KT, Lk - j0);
  if (nkeys <= 0) return;
  const int off = Lk - Lq;
  const int pos_hi = a.window > 0 ? min(Lk - 1, j0 + nkeys - 1 + a.window - 1) : Lk - 1;
  const int t_lo = max(0, j0 - off), t_hi = min(Lq - 1, pos_hi - off);
  const int qt_lo = t_lo / QT, n_qt = t_hi >= t_lo ? t_hi / QT - qt_lo + 1 : 0;
  const int nsteps = hpc * n_qt;
  const bool has_bias = a.rd > 0 && a.E > 0;
  auto step_h = [&](int n) { return g * a.group + half * hpc + n / n_qt; };
  auto step_t0 = [&](int n) { return (qt_lo + n % n_qt) * QT; };
  auto is_band = [&](int t0) { return has_bias && (off + t0 - (j0 + KT - 1) < a.E); };

  // ------------------------------------------------------------ set-up
  if (tid == 0) {
    mbar_init(bar(B_KV_FULL), 1);
    for (int s = 0; s < QSTAGES; ++s) {
      mbar_init(bar(B_Q_FULL + s), 1);
      mbar_init(bar(B_Q_EMPTY + s), 1);
      mbar_init(bar(B_AUX_FULL + s), 32);
      mbar_init(bar(B_AUX_EMPTY + s), NELEM);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_S_FULL + i), 1);
      mbar_init(bar(B_P_FULL + i), NELEM);
    }
    mbar_init(bar(B_R_FULL), 1);
    mbar_init(bar(B_RW_READ), NELEM);
    mbar_init(bar(B_DONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + SM_TMEM_SLOT, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map_k);
    prefetch_tmap(&map_v);
    prefetch_tmap(&map_q);
    prefetch_tmap(&map_do);
    if (a.rd > 0 && a.E > 0) prefetch_tmap(&map_r);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + SM_TMEM_SLOT);

  if (warp == 0) {
    // ======================================================== TMA producer
    if (lane == 0) {
      bool run = true;
      int issued = 0;
      mbar_arrive_expect_tx(bar(B_KV_FULL), 65536);
      tma_load_3d(sb + SM_K, &map_k, 0, g, ck + j0, bar(B_KV_FULL));
      tma_load_3d(sb + SM_K + 16384, &map_k, 64, g, ck + j0, bar(B_KV_FULL));
      tma_load_3d(sb + SM_V, &map_v, 0, g, ck + j0, bar(B_KV_FULL));
      tma_load_3d(sb + SM_V + 16384, &map_v, 64, g, ck + j0, bar(B_KV_FULL));
      for (int n = 0; n < nsteps && run; ++n) {
        const int st = n % QSTAGES;
        if (n >= QSTAGES &&
            !(run = mbar_wait(bar(B_Q_EMPTY + st), ((n / QSTAGES) - 1) & 1, abort_flag, 1)))
          break;
        const int h = step_h(n), row = cq + step_t0(n);
        const uint32_t dq = sb + SM_Q + st * 16384, dd = sb + SM_DO + st * 16384;
        if (n != a.test_skip_dkdv_step) {   // (test hook: a skipped step is never loaded)
          mbar_arrive_expect_tx(bar(B_Q_FULL + st), 32768);
          tma_load_3d(dq, &map_q, 0, h, row, bar(B_Q_FULL + st));
          tma_load_3d(dq + 8192, &map_q, 64, h, row, bar(B_Q_FULL + st));
          tma_load_3d(dd, &map_do, 0, h, row, bar(B_Q_FULL + st));
          tma_load_3d(dd + 8192, &map_do, 64, h, row, bar(B_Q_FULL + st));
        }
        issued = n + 1;
      }
      if (*abort_flag) {   // let the copies this thread issued land before the CTA exits
        drain_wait(bar(B_KV_FULL), 0);
        for (int m = max(0, issued - QSTAGES); m < issued; ++m)
          drain_wait(bar(B_Q_FULL + m % QSTAGES), (m / QSTAGES) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================================================== MMA issuer
    // The whole warp runs the issue code (descriptors stay warp-uniform); each
    // MMA and commit is issued by one elected lane.
    {
      bool ok = mbar_wait_warp(bar(B_KV_FULL), 0, abort_flag, 2);
      tc_fence_after();
      const uint32_t id_s = idesc_bf16_f32(KT, QT, 0, 0);    // S^T: K (smem, K-major) x Q (smem, K-major)
      const uint32_t id_o = idesc_bf16_f32(KT, 128, 0, 1);   // dV: P^T (tmem) x dout (smem, MN-major)
      const uint64_t kd = smem_desc_sw128(sb + SM_K, 16, 1024);
      const uint64_t vd = smem_desc_sw128(sb + SM_V, 16, 1024);
      for (int n = 0; n <= nsteps && ok; ++n) {
        if (n < nsteps) {
          const int st = n % QSTAGES, buf = n & 1;
          if (!(ok = mbar_wait_warp(bar(B_Q_FULL + st), (n / QSTAGES) & 1, abort_flag, 3))) break;
          tc_fence_after();
          const uint64_t qd = smem_desc_sw128(sb + SM_Q + st * 16384, 16, 1024);
          const uint64_t dd = smem_desc_sw128(sb + SM_DO + st * 16384, 16, 1024);
          const uint32_t d_s = tmem + TM_ST + 64u * buf, d_p = tmem + TM_DP + 64u * buf;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // 16 dims a step: 32 bytes into a 128-byte row; the second 64 dims are
            // the second box (K / V: 16 KB on, q / dout: 8 KB on)
            const uint32_t ad = kk < 4 ? 2u * kk : 1024u + 2u * (kk - 4);
            const uint32_t bd = kk < 4 ? 2u * kk : 512u + 2u * (kk - 4);
            mma_ss_e(d_s, kd + ad, qd + bd, id_s, kk > 0);
            mma_ss_e(d_p, vd + ad, dd + bd, id_s, kk > 0);
          }
          mma_commit_e(bar(B_S_FULL + buf));
        }
        if (n >= 1) {
          const int m = n - 1, st = m % QSTAGES, buf = m & 1;
          if (!(ok = mbar_wait_warp(bar(B_P_FULL + buf), (m >> 1) & 1, abort_flag, 4))) break;
          tc_fence_after();
          const uint32_t pa = tmem + TM_ST + 64u * buf, sa = tmem + TM_DP + 64u * buf;
          // MN-major q / dout: 16 query rows a step (2 KB), the two 64-dim boxes 8 KB apart
          const uint64_t om = smem_desc_sw128(sb + SM_DO + st * 16384, 8192, 1024);
          const uint64_t qm = smem_desc_sw128(sb + SM_Q + st * 16384, 8192, 1024);
#pragma unroll
          for (int kq = 0; kq < QT / 16; ++kq) {
            const uint32_t acc = (m > 0 || kq > 0) ? 1u : 0u;
            const uint32_t ac = 8u * kq + (kq >= 2 ? 16u : 0u);   // P^T / dS^T columns: [0,16) [32,48)
            mma_ts_e(tmem + TM_DV, pa + ac, om + 128u * kq, id_o, acc);
            mma_ts_e(tmem + TM_DK, sa + ac, qm + 128u * kq, id_o, acc);
          }
          mma_commit_e(bar(B_Q_EMPTY + st));   // the stage's q / dout have been read
        }
      }
      if (ok) {
        mma_commit_e(bar(B_DONE));
      } else {
        // stop: wait for the MMAs already issued before tensor memory is freed
        mma_commit_e(bar(B_DRAIN));
        drain_wait(bar(B_DRAIN), 0);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ======================================================== per-step constants and R windows
    // One warp, so that its only synchronisation is __syncwarp (a wait that
    // gives up can never leave another warp stuck at a barrier).
    int nb = 0;                          // band steps so far
    int issued_r = 0;                    // (lane 0) R windows requested
    bool run = true;
    for (int n = 0; n < nsteps && run; ++n) {
      const int st = n % QSTAGES;
      if (n >= QSTAGES && !(run = mbar_wait(bar(B_AUX_EMPTY + st), ((n / QSTAGES) - 1) & 1, abort_flag, 5)))
        break;
      const int h = step_h(n), t0 = step_t0(n);
      float *ax = reinterpret_cast<float *>(smem + SM_AUX + st * 4 * QT * 4);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int at = lane + 32 * e, t = t0 + at;
        const bool okr = t < Lq;
        const size_t li = (size_t)h * a.total_q + cq + (okr ? t : 0);
        const float sc = log_scale(off + t, a.inv_ln_base);
        ax[at] = okr ? a.lse[li] * kLog2e : INFINITY;
        ax[QT + at] = okr ? a.Dsum[li] : 0.f;
        ax[2 * QT + at] = sc * kLog2e;
        ax[3 * QT + at] = sc * a.alpha;
      }
      mbar_arrive(bar(B_AUX_FULL + st));
      if (!is_band(t0)) continue;
      // the R window of this band step: R rows t0 .. t0 + 63 of head h,
      // distances cb .. cb + 199 (negative distances and those past E read as
      // zero: the box starts left of / runs past the tensor)
      if (nb > 0 && !(run = mbar_wait(bar(B_RW_READ), (nb - 1) & 1, abort_flag, 6))) break;
      if (lane == 0) {
        const int cb = floor8(off + t0 - (j0 + KT - 1));
        mbar_arrive_expect_tx(bar(B_R_FULL), QT * RWC * 4);
        tma_load_3d(sb + SM_RW, &map_r, cb, h, cq + t0, bar(B_R_FULL));
        issued_r = nb + 1;
      }
      ++nb;
    }
    if (*abort_flag && lane == 0 && issued_r > 0) drain_wait(bar(B_R_FULL), (issued_r - 1) & 1);
  } else if (warp >= 4) {
    // ======================================================== elementwise
    // Warp 4 + q + 4 hh (q = warp & 3) takes TMEM lanes 32 q .. 32 q + 31 (one
    // key row a thread) and query columns 32 hh .. 32 hh + 31 of each step;
    // its P^T / dS^T go to columns [32 hh, 32 hh + 16), which hold S^T / dP^T
    // values this same warp has already read (the other warp of the row
    // reads its own 32 columns whenever it gets there).
    const int hh = (warp - 4) >> 2;
    const int jl = 32 * (warp & 3) + lane;             // key row = TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const int j = j0 + jl;
    int nb = 0;
    bool ok = true;
    for (int n = 0; n < nsteps && ok; ++n) {
      const int st = n % QSTAGES, buf = n & 1;
      const int t0 = step_t0(n), pos0 = off + t0;
      const bool band = is_band(t0);
      const int cb = floor8(pos0 - (j0 + KT - 1));
      ok = mbar_wait(bar(B_S_FULL + buf), (n >> 1) & 1, abort_flag, 7) &&
           mbar_wait(bar(B_AUX_FULL + st), (n / QSTAGES) & 1, abort_flag, 8) &&
           (!band || mbar_wait(bar(B_R_FULL), nb & 1, abort_flag, 9));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float *ax = reinterpret_cast<const float *>(smem + SM_AUX + st * 4 * QT * 4);
      const float *rw = reinterpret_cast<const float *>(smem + SM_RW);
      const bool need_mask = (j0 + KT - 1 > pos0) || (a.window > 0 && j0 < pos0 + QT - 1 - a.window + 1);
      uint32_t sv[32], dv[32];
      tmem_ld32(tmem + lane_off + TM_ST + 64u * buf + 32u * hh, sv);
      tmem_ld32(tmem + lane_off + TM_DP + 64u * buf + 32u * hh, dv);
      tmem_wait_ld();
      // alpha S^T + bias for this thread's 32 query rows, the bias gathered
      // from the window at once, so the window is released (and the next
      // band step's copy can start) before the rest of the step's work
      if (band) {
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int i = 32 * hh + u;
          sv[u] = __float_as_uint(fmaf(__uint_as_float(sv[u]), a.alpha, rw[i * RWS + (pos0 + i - j - cb)]));
        }
        mbar_arrive(bar(B_RW_READ));   // this thread has gathered from the window
        ++nb;
      } else {
#pragma unroll
        for (int u = 0; u < 32; ++u) sv[u] = __float_as_uint(__uint_as_float(sv[u]) * a.alpha);
      }
      uint32_t pk[16], dk2[16];
#pragma unroll
      for (int u = 0; u < 32; u += 4) {
        const int i0 = 32 * hh + u;                    // 4 query rows of the step
        const float4 l4 = *reinterpret_cast<const float4 *>(ax + i0);
        const float4 d4 = *reinterpret_cast<const float4 *>(ax + QT + i0);
        const float4 c4 = *reinterpret_cast<const float4 *>(ax + 2 * QT + i0);
        const float4 a4 = *reinterpret_cast<const float4 *>(ax + 3 * QT + i0);
        const float lse2[4] = {l4.x, l4.y, l4.z, l4.w}, Di[4] = {d4.x, d4.y, d4.z, d4.w};
        const float c1[4] = {c4.x, c4.y, c4.z, c4.w}, c3[4] = {a4.x, a4.y, a4.z, a4.w};
        float pv[4], dsv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pos = pos0 + i0 + e;
          float x = __uint_as_float(sv[u + e]) * c1[e];
          if (need_mask) {
            const bool vis = j <= pos && (a.window <= 0 || pos - j < a.window);
            if (!vis) x = -INFINITY;
          }
          const float p = fast_exp2(x - lse2[e]);
          pv[e] = p;
          dsv[e] = p * (__uint_as_float(dv[u + e]) - Di[e]) * c3[e];
        }
        pk[(u >> 1)] = pack_bf16x2(pv[0], pv[1]);
        pk[(u >> 1) + 1] = pack_bf16x2(pv[2], pv[3]);
        dk2[(u >> 1)] = pack_bf16x2(dsv[0], dsv[1]);
        dk2[(u >> 1) + 1] = pack_bf16x2(dsv[2], dsv[3]);
      }
      tmem_st16(tmem + lane_off + TM_ST + 64u * buf + 32u * hh, pk);   // P^T
      tmem_st16(tmem + lane_off + TM_DP + 64u * buf + 32u * hh, dk2);  // dS^T
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_P_FULL + buf));
      mbar_arrive(bar(B_AUX_EMPTY + st));
    }
    // ---- dK / dV rows out (zeros when no query sees the keys); the TMEM
    // loads are warp-collective, the stores only for rows inside the keys
    if (ok && (nsteps == 0 || mbar_wait(bar(B_DONE), 0, abort_flag, 10))) {
      tc_fence_after();
      const size_t row = (size_t)(ck + j) * a.Hkv + g;
      {
        const int which = hh;                          // hh 0: dK, hh 1: dV
        __nv_bfloat16 *dst = (which ? a.dv : a.dk) + row * kHeadDim;
        // with a split: this half's fp32 sums, added by relattn_bwd_dkv_reduce_kernel
        float *pdst = a.kv_split > 1 ? a.dkv_part + ((size_t)(2 * half + which) * a.total_k * a.Hkv + row) * kHeadDim
                                     : nullptr;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          if (nsteps > 0) {
            tmem_ld32(tmem + lane_off + (which ? TM_DV : TM_DK) + 32u * c, v);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
          }
          if (jl < nkeys && pdst) {
            float4 *d4 = reinterpret_cast<float4 *>(pdst + 32 * c);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              d4[q4] = make_float4(__uint_as_float(v[4 * q4]), __uint_as_float(v[4 * q4 + 1]),
                                   __uint_as_float(v[4 * q4 + 2]), __uint_as_float(v[4 * q4 + 3]));
          } else if (jl < nkeys) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 o;
              o.x = pack_bf16x2(__uint_as_float(v[8 * q4 + 0]), __uint_as_float(v[8 * q4 + 1]));
              o.y = pack_bf16x2(__uint_as_float(v[8 * q4 + 2]), __uint_as_float(v[8 * q4 + 3]));
              o.z = pack_bf16x2(__uint_as_float(v[8 * q4 + 4]), __uint_as_float(v[8 * q4 + 5]));
              o.w = pack_bf16x2(__uint_as_float(v[8 * q4 + 6]), __uint_as_float(v[8 * q4 + 7]));
              *reinterpret_cast<uint4 *>(dst + 32 * c + 8 * q4) = o;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) record_timeout(a.err, *abort_flag);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}


// dk / dv = the two halves' fp32 sums, in bf16 (a split dk / dv launch).  A
// warp per key row.  Only rows the split dk / dv CTAs wrote are touched: rows
// of sequences with consistent lengths, below cu_seqlens_k[batch] (rows past
// it, and the rows of a sequence the kernels skipped, keep their contents, as
// on the unsplit path).
__global__ void __launch_bounds__(256) relattn_bwd_dkv_reduce_kernel(const BwdArgs a) {
  const size_t n4 = (size_t)a.total_k * a.Hkv * (kHeadDim / 4);   // float4 groups per tensor
  const float4 *p = reinterpret_cast<const float4 *>(a.dkv_part);
  const int lane = threadIdx.x & 31;
  const int rows = min(a.cu_k[a.batch], a.total_k);
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nwarps) {
    int lo = 0, hi = a.batch - 1;                  // the sequence of key row r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.cu_k[mid] <= r) lo = mid;
      else hi = mid - 1;
    }
    const int Lq = a.cu_q[lo + 1] - a.cu_q[lo], Lk = a.cu_k[lo + 1] - a.cu_k[lo];
    if (r < a.cu_k[lo] || Lq < 0 || Lk < Lq || Lq > a.max_q || Lk > a.max_k) continue;
    for (int h = 0; h < a.Hkv; ++h) {
      const size_t k = ((size_t)r * a.Hkv + h) * (kHeadDim / 4) + lane;
#pragma unroll
      for (int which = 0; which < 2; ++which) {                   // 0: dk, 1: dv
        const float4 x = p[which * n4 + k], y = p[(2 + which) * n4 + k];
        uint2 o;
        o.x = pack_bf16x2(x.x + y.x, x.y + y.y);
        o.y = pack_bf16x2(x.z + y.z, x.w + y.w);
        *reinterpret_cast<uint2 *>((which ? a.dv : a.dk) + 4 * k) = o;
      }
    }
  }
}

// ====================================================================== dq (query-major)
//
// For 128 query rows of one head and the 128-key steps every row of the
// tile sees outside the bias band (j < kend, kend = p0 - E + 1 rounded down
// to a multiple of 64 for the tile's first position p0, so no bias and no
// dr; every visible key without a bias):
//     S = Q K^T,  dP = dout V^T                          (tcgen05, M = 128 rows, N = 128 keys)
//     P = exp(s_i alpha S - lse_i),  dS' = s_i P (dP - D_i)
//     dQ += dS' K                                          (tcgen05, A = dS' in TMEM)
// and dq = alpha dQ.  Roles as in the dk / dv kernel, without the aux warp:
// each elementwise thread owns one query row, so its constants stay in
// registers.  128-key steps: an N = 128 instruction costs about what an
// N = 64 one does to issue, so S and dP take half the instructions per key.
// TMEM: dQ [0,128), S buffers [128,256) / [256,384) (dS' as bf16 pairs over
// columns [0,32) and [64,96) of its buffer: each elementwise warp packs its
// 64 keys over the first half of the columns it has read), one dP buffer
// [384,512): dP of step n+1 is issued once every elementwise thread has
// loaded dP of step n (D_DP_READ), early in that thread's step.
constexpr int QM = 128;          // query rows per CTA (MMA M)
constexpr int KS = 128;          // keys per step (MMA N of S / dP, K of dQ)
constexpr int KSTAGES = 2;
constexpr uint32_t TQ_DQ = 0, TQ_S = 128, TQ_DP = 384;
constexpr uint32_t SQ_Q = 0;                            // 2 boxes [128 rows x 128 B]
constexpr uint32_t SQ_DO = SQ_Q + 32768;
constexpr uint32_t SQ_K = SQ_DO + 32768;                // KSTAGES x 2 boxes [128 keys x 128 B]
constexpr uint32_t SQ_V = SQ_K + KSTAGES * 32768;
constexpr uint32_t SQ_BAR = SQ_V + KSTAGES * 32768;
enum {
  D_QD_FULL = 0,
  D_KV_FULL = 1,                      // + stage
  D_KV_EMPTY = D_KV_FULL + KSTAGES,   // + stage
  D_S_FULL = D_KV_EMPTY + KSTAGES,    // + buffer
  D_P_FULL = D_S_FULL + 2,            // + buffer
  D_DP_READ = D_P_FULL + 2,
  D_DONE = D_DP_READ + 1,
  D_DRAIN = D_DONE + 1,
  D_COUNT = D_DRAIN + 1
};
constexpr uint32_t SQ_TMEM_SLOT = SQ_BAR + D_COUNT * 8;
constexpr uint32_t SQ_ABORT = SQ_TMEM_SLOT + 8;
constexpr uint32_t SQ_TOTAL = SQ_ABORT + 8;
constexpr uint32_t SMEM_BYTES_DQ = SQ_TOTAL + 1024;
static_assert(SMEM_BYTES_DQ <= 227 * 1024, "shared memory budget");

__global__ void __launch_bounds__(NTHR, 1)
relattn_bwd_dq_tc_kernel(const __grid_constant__ BwdArgs a,
                         const __grid_constant__ CUtensorMap map_q,
                         const __grid_constant__ CUtensorMap map_do,
                         const __grid_constant__ CUtensorMap map_k,
                         const __grid_constant__ CUtensorMap map_v) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sb = smem_addr(smem);
  auto bar = [&](int i) { return sb + SQ_BAR + 8u * i; };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SQ_ABORT);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ------------------------------------------------------------ the CTA's rows and key steps
  const int h = blockIdx.y, b = blockIdx.z, g = h / a.group;
  const int cq = a.cu_q[b], ck = a.cu_k[b];
  const int Lq = a.cu_q[b + 1] - cq, Lk = a.cu_k[b + 1] - ck;
  if (Lq < 0 || Lk < Lq || Lq > a.max_q || Lk > a.max_k) {
    if (tid == 0) atomicOr(a.err, kDevErrSeqlens);
    return;
  }
  const int row0 = (int)(gridDim.x - 1 - blockIdx.x) * QM;   // longest first
  const int nrows = min(QM, Lq - row0);
  if (nrows <= 0) return;
  const int off = Lk - Lq;
  const int p0 = off + row0, p_end = p0 + nrows - 1;
  const int j_lo = a.window > 0 ? max(0, p0 - a.window + 1) : 0;
  const int kbeg = j_lo & ~(KS - 1);
  const bool has_bias = a.rd > 0 && a.E > 0;
  // without a bias every visible key; with one, the keys below the band of
  // the tile's first row (a multiple of 64: the warp-MMA dq starts there);
  // keys of the last step at or past kend are masked out
  const int kend = has_bias ? (p0 - a.E + 1 > 0 ? (p0 - a.E + 1) & ~63 : 0) : p_end + 1;
  const int nsteps = kend > kbeg ? (kend - kbeg + KS - 1) / KS : 0;

  // ------------------------------------------------------------ set-up
  if (tid == 0) {
    mbar_init(bar(D_QD_FULL), 1);
    for (int s = 0; s < KSTAGES; ++s) {
      mbar_init(bar(D_KV_FULL + s), 1);
      mbar_init(bar(D_KV_EMPTY + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(D_S_FULL + i), 1);
      mbar_init(bar(D_P_FULL + i), NELEM);
    }
    mbar_init(bar(D_DP_READ), NELEM);
    mbar_init(bar(D_DONE), 1);
    mbar_init(bar(D_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + SQ_TMEM_SLOT, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map_q);
    prefetch_tmap(&map_do);
    prefetch_tmap(&map_k);
    prefetch_tmap(&map_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + SQ_TMEM_SLOT);

  if (warp == 0) {
    // ======================================================== TMA producer
    if (lane == 0 && nsteps > 0) {
      bool run = true;
      int issued = 0;
      mbar_arrive_expect_tx(bar(D_QD_FULL), 65536);
      tma_load_3d(sb + SQ_Q, &map_q, 0, h, cq + row0, bar(D_QD_FULL));
      tma_load_3d(sb + SQ_Q + 16384, &map_q, 64, h, cq + row0, bar(D_QD_FULL));
      tma_load_3d(sb + SQ_DO, &map_do, 0, h, cq + row0, bar(D_QD_FULL));
      tma_load_3d(sb + SQ_DO + 16384, &map_do, 64, h, cq + row0, bar(D_QD_FULL));
      for (int n = 0; n < nsteps && run; ++n) {
        const int st = n % KSTAGES;
        if (n >= KSTAGES &&
            !(run = mbar_wait(bar(D_KV_EMPTY + st), ((n / KSTAGES) - 1) & 1, abort_flag, 11)))
          break;
        const int key = ck + kbeg + n * KS;
        const uint32_t dk_ = sb + SQ_K + st * 32768, dv_ = sb + SQ_V + st * 32768;
        if (n != a.test_skip_dq_step) {   // (test hook: a skipped step is never loaded)
          mbar_arrive_expect_tx(bar(D_KV_FULL + st), 65536);
          tma_load_3d(dk_, &map_k, 0, g, key, bar(D_KV_FULL + st));
          tma_load_3d(dk_ + 16384, &map_k, 64, g, key, bar(D_KV_FULL + st));
          tma_load_3d(dv_, &map_v, 0, g, key, bar(D_KV_FULL + st));
          tma_load_3d(dv_ + 16384, &map_v, 64, g, key, bar(D_KV_FULL + st));
        }
        issued = n + 1;
      }
      if (*abort_flag) {   // let the copies this thread issued land before the CTA exits
        drain_wait(bar(D_QD_FULL), 0);
        for (int m = max(0, issued - KSTAGES); m < issued; ++m)
          drain_wait(bar(D_KV_FULL + m % KSTAGES), (m / KSTAGES) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================================================== MMA issuer
    // The whole warp runs the issue code (descriptors stay warp-uniform); each
    // MMA and commit is issued by one elected lane.
    if (nsteps > 0) {
      bool ok = mbar_wait_warp(bar(D_QD_FULL), 0, abort_flag, 12);
      tc_fence_after();
      const uint32_t id_s = idesc_bf16_f32(QM, KS, 0, 0);    // S: Q (smem, K-major) x K (smem, K-major)
      const uint32_t id_o = idesc_bf16_f32(QM, 128, 0, 1);   // dQ: dS' (tmem) x K (smem, MN-major)
      const uint64_t qd = smem_desc_sw128(sb + SQ_Q, 16, 1024);
      const uint64_t dd = smem_desc_sw128(sb + SQ_DO, 16, 1024);
      for (int n = 0; n <= nsteps && ok; ++n) {
        if (n < nsteps) {
          // S(n) into buffer n & 1 (the dQ MMA of step n - 2, which read its
          // dS', was issued before); dP(n) once dP(n - 1) has been loaded
          const int st = n % KSTAGES, buf = n & 1;
          if (!(ok = mbar_wait_warp(bar(D_KV_FULL + st), (n / KSTAGES) & 1, abort_flag, 13))) break;
          tc_fence_after();
          const uint64_t kd = smem_desc_sw128(sb + SQ_K + st * 32768, 16, 1024);
          const uint64_t vd = smem_desc_sw128(sb + SQ_V + st * 32768, 16, 1024);
          const uint32_t d_s = tmem + TQ_S + 128u * buf, d_p = tmem + TQ_DP;
          // 16 dims a step: 32 bytes into a 128-byte row; the second 64 dims are
          // the second box (16 KB on for Q / dout and for K / V)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ad = kk < 4 ? 2u * kk : 1024u + 2u * (kk - 4);
            mma_ss_e(d_s, qd + ad, kd + ad, id_s, kk > 0);
          }
          if (n >= 1 && !(ok = mbar_wait_warp(bar(D_DP_READ), (n - 1) & 1, abort_flag, 17))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ad = kk < 4 ? 2u * kk : 1024u + 2u * (kk - 4);
            mma_ss_e(d_p, dd + ad, vd + ad, id_s, kk > 0);
          }
          mma_commit_e(bar(D_S_FULL + buf));
        }
        if (n >= 1) {
          const int m = n - 1, st = m % KSTAGES, buf = m & 1;
          if (!(ok = mbar_wait_warp(bar(D_P_FULL + buf), (m >> 1) & 1, abort_flag, 14))) break;
          tc_fence_after();
          const uint32_t pa = tmem + TQ_S + 128u * buf;
          // MN-major K: 16 keys a step (2 KB), the two 64-dim boxes 16 KB apart
          const uint64_t km = smem_desc_sw128(sb + SQ_K + st * 32768, 16384, 1024);
#pragma unroll
          for (int kq = 0; kq < KS / 16; ++kq)   // dS' columns: [0,32) keys 0..63, [64,96) keys 64..127
            mma_ts_e(tmem + TQ_DQ, pa + 8u * kq + (kq >= 4 ? 32u : 0u), km + 128u * kq, id_o,
                   (m > 0 || kq > 0) ? 1u : 0u);
          mma_commit_e(bar(D_KV_EMPTY + st));   // the stage's K / V have been read
        }
      }
      if (ok) {
        mma_commit_e(bar(D_DONE));
      } else {
        mma_commit_e(bar(D_DRAIN));
        drain_wait(bar(D_DRAIN), 0);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ======================================================== elementwise
    // Warp 4 + q + 4 hh (q = warp & 3) takes TMEM lanes 32 q .. 32 q + 31 (one
    // query row a thread) and keys 64 hh .. 64 hh + 63 of each step, in two
    // halves of 32; its dS' goes to columns [64 hh, 64 hh + 32) of the S
    // buffer, which hold S values this same warp has already read.
    const int hh = (warp - 4) >> 2;
    const int il = 32 * (warp & 3) + lane;             // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const int t = row0 + il, pos = off + t;
    const bool okr = il < nrows;
    const size_t li = (size_t)h * a.total_q + cq + (okr ? t : 0);
    const float srow = log_scale(pos, a.inv_ln_base);
    const float c1 = a.alpha_log2e * srow;
    const float lse2 = okr ? a.lse[li] * kLog2e : INFINITY;   // rows past the end: P = 0
    const float Di = okr ? a.Dsum[li] : 0.f;
    bool ok = true;
    for (int n = 0; n < nsteps && ok; ++n) {
      const int buf = n & 1, j0 = kbeg + n * KS;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(D_S_FULL + buf), (n >> 1) & 1, abort_flag, 15));
      if (!ok) break;
      tc_fence_after();
      const bool need_mask =
          (j0 + KS - 1 > p0) || (a.window > 0 && j0 < p_end - a.window + 1) || (j0 + KS > kend);
      const uint32_t sbuf = tmem + lane_off + TQ_S + 128u * buf + 64u * hh;
      uint32_t sv[32], dv[2][32];
      tmem_ld32(tmem + lane_off + TQ_DP + 64u * hh, dv[0]);
      tmem_ld32(tmem + lane_off + TQ_DP + 64u * hh + 32u, dv[1]);
      tmem_ld32(sbuf, sv);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(D_DP_READ));   // dP(n) is in registers: dP(n + 1) may be written
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (c == 1) {
          tmem_ld32(sbuf + 32u, sv);
          tmem_wait_ld();
        }
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
          float d2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float x = __uint_as_float(sv[u + e]) * c1;
            if (need_mask) {
              const int j = j0 + 64 * hh + 32 * c + u + e;
              const bool vis = j <= pos && j < kend && (a.window <= 0 || pos - j < a.window);
              if (!vis) x = -INFINITY;
            }
            const float p = fast_exp2(x - lse2);
            d2[e] = p * (__uint_as_float(dv[c][u + e]) - Di) * srow;
          }
          pk[u >> 1] = pack_bf16x2(d2[0], d2[1]);
        }
        tmem_st16(sbuf + 16u * c, pk);   // dS' over S columns this warp has read
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(D_P_FULL + buf));
    }
    // ---- dq rows out: alpha dQ, fp32 into the workspace when the band's
    // kernel adds to it, else bf16; hh 0 takes columns 0..63, hh 1 64..127
    if (ok && (nsteps == 0 || mbar_wait(bar(D_DONE), 0, abort_flag, 16))) {
      tc_fence_after();
      const size_t row = (size_t)(cq + t) * a.Hq + h;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        const int col = 64 * hh + 32 * c;
        uint32_t v[32];
        if (nsteps > 0) {
          tmem_ld32(tmem + lane_off + TQ_DQ + (uint32_t)col, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (!okr) continue;
        if (a.dq_split) {
          float4 *dst = reinterpret_cast<float4 *>(a.dq_part + row * kHeadDim + col);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            dst[q4] = make_float4(__uint_as_float(v[4 * q4]) * a.alpha, __uint_as_float(v[4 * q4 + 1]) * a.alpha,
                                  __uint_as_float(v[4 * q4 + 2]) * a.alpha, __uint_as_float(v[4 * q4 + 3]) * a.alpha);
        } else {
          __nv_bfloat16 *dst = a.dq + row * kHeadDim + col;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(v[8 * q4 + 0]) * a.alpha, __uint_as_float(v[8 * q4 + 1]) * a.alpha);
            o.y = pack_bf16x2(__uint_as_float(v[8 * q4 + 2]) * a.alpha, __uint_as_float(v[8 * q4 + 3]) * a.alpha);
            o.z = pack_bf16x2(__uint_as_float(v[8 * q4 + 4]) * a.alpha, __uint_as_float(v[8 * q4 + 5]) * a.alpha);
            o.w = pack_bf16x2(__uint_as_float(v[8 * q4 + 6]) * a.alpha, __uint_as_float(v[8 * q4 + 7]) * a.alpha);
            *reinterpret_cast<uint4 *>(dst + 8 * q4) = o;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) record_timeout(a.err, *abort_flag);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}
}  // namespace

namespace {

PFN_cuTensorMapEncodeTiled_v12000 bwd_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [rows, heads, 128] bf16 in boxes of 64 dims x 1 head x box_rows rows, 128-byte swizzle
bool encode_rows(CUtensorMap *m, const void *base, int heads, int rows, int box_rows) {
  auto fn = bwd_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {256, (cuuint64_t)heads * 256};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool bwd_tc_supported(const BwdArgs &a) {
  auto al = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!bwd_encoder()) return false;
  if (!al(a.q) || !al(a.k) || !al(a.v) || !al(a.dout)) return false;
  if (a.rd_pad > 64) return false;
  return a.total_k >= KT && a.total_q >= QT;   // the TMA boxes stay inside the tensors
}

cudaError_t launch_bwd_dkdv_tc(const BwdArgs &a, cudaStream_t stream) {
  CUtensorMap mk, mv, mq, md, mr;
  if (!encode_rows(&mk, a.k, a.Hkv, a.total_k, KT) || !encode_rows(&mv, a.v, a.Hkv, a.total_k, KT) ||
      !encode_rows(&mq, a.q, a.Hq, a.total_q, QT) || !encode_rows(&md, a.dout, a.Hq, a.total_q, QT))
    return cudaErrorInvalidValue;
  mr = mk;   // (unused without a bias)
  if (a.rd > 0 && a.E > 0) {
    // R [Tq, Hq, e_pad] fp32 in boxes of 200 distances x 1 head x 64 rows, no swizzle
    cuuint64_t dims[3] = {(cuuint64_t)a.E, (cuuint64_t)a.Hq, (cuuint64_t)a.total_q};
    cuuint64_t strides[2] = {(cuuint64_t)a.e_pad * 4, (cuuint64_t)a.Hq * a.e_pad * 4};
    cuuint32_t box[3] = {(cuuint32_t)RWC, 1, (cuuint32_t)QT};
    cuuint32_t es[3] = {1, 1, 1};
    auto fn = bwd_encoder();
    if (!fn || fn(&mr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.Rall, dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  static std::atomic<bool> attr_set[kMaxDevicesAttr];
  {
    cudaError_t e = set_max_smem_once(reinterpret_cast<const void *>(relattn_bwd_dkdv_tc_kernel),
                                      (int)SMEM_BYTES_BWD, attr_set);
    if (e != cudaSuccess) return e;
  }
  // An even GQA group of at least 4 heads is split between two CTAs per key
  // tile: twice the CTAs, half the longest one (the last wave is the ragged
  // part of this grid), and one small reduce launch.
  BwdArgs ak = a;
  ak.kv_split = (a.dkv_part != nullptr && a.group >= 4 && a.group % 2 == 0) ? 2 : 1;
  const int k_tiles = (a.max_k + KT - 1) / KT;
  relattn_bwd_dkdv_tc_kernel<<<dim3(k_tiles, a.Hkv * ak.kv_split, a.batch), NTHR, SMEM_BYTES_BWD, stream>>>(
      ak, mk, mv, mq, md, mr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || ak.kv_split == 1) return e;
  // a warp per key row, 8 rows per CTA, grid-stride beyond 8 CTAs per SM
  const unsigned blocks = (unsigned)std::min<size_t>(((size_t)a.total_k + 7) / 8, 152 * 8);
  if (blocks > 0) relattn_bwd_dkv_reduce_kernel<<<blocks, 256, 0, stream>>>(ak);
  return cudaGetLastError();
}

bool bwd_dq_tc_supported(const BwdArgs &a) {
  return bwd_tc_supported(a) && a.total_q >= QM && a.total_k >= KS;   // the TMA boxes stay inside
}

cudaError_t launch_bwd_dq_tc(const BwdArgs &a, cudaStream_t stream) {
  CUtensorMap mq, md, mk, mv;
  if (!encode_rows(&mq, a.q, a.Hq, a.total_q, QM) || !encode_rows(&md, a.dout, a.Hq, a.total_q, QM) ||
      !encode_rows(&mk, a.k, a.Hkv, a.total_k, KS) || !encode_rows(&mv, a.v, a.Hkv, a.total_k, KS))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[kMaxDevicesAttr];
  {
    cudaError_t e = set_max_smem_once(reinterpret_cast<const void *>(relattn_bwd_dq_tc_kernel),
                                      (int)SMEM_BYTES_DQ, attr_set);
    if (e != cudaSuccess) return e;
  }
  const int q_tiles = (a.max_q + QM - 1) / QM;
  relattn_bwd_dq_tc_kernel<<<dim3(q_tiles, a.Hq, a.batch), NTHR, SMEM_BYTES_DQ, stream>>>(a, mq, md, mk, mv);
  return cudaGetLastError();
}

}  // namespace relattn
