// fwd_tc_main.cu -- relative-attention prefill on 5th-generation tensor cores,
// the key tiles outside the relative-bias band (all of them when there is no
// bias).  Same computation as the definition on the page "SGLang and Miles Add
// Day-0 Support for Inkling", section "Attention with Relative Positional
// Embedding": past the band, x(i,j) = s(i) * alpha * q_i.k_j.
//
// One CTA = 128 query rows x two query heads of the same GQA group, so the two
// heads share every K/V tile and every mask.  Warp roles:
//   warp 0      TMA producer (one thread): the two Q tiles once, then K and V
//               tiles of 128 keys (2- and 3-stage rings)
//   warp 1      TMEM allocator; MMA issuer (the whole warp runs the issue
//               code, an elected lane issues): S_w = Q_w K^T (both operands in
//               shared memory), O_w += P_w V (P_w in TMEM)
//   warps 2-3   idle
//   warps 4-7   softmax of head 0, warps 8-11 softmax of head 1: thread = row,
//               all 128 keys of a tile
// The issuer alternates the heads (S0, S1, PV0, S0', PV1, S1', ...): while one
// head's softmax runs, the tensor core works for the other.
//
// Tensor memory: O0 [0,128), O1 [128,256), S0 [256,384), S1 [384,512); head
// w's P (bf16) is written over the first 64 columns of S_w.
//
// When the band was done first (by the bias kernel, which leaves out / lse
// normalised over the band keys), each row starts from that state:
// m = lse * log2(e), l = 1, O = out -- the online softmax carried over.
//
// Every wait is bounded; a timeout sets the device error word, the CTA drains
// its own copies / MMAs with bounded waits, frees TMEM and exits.
#include <cudaTypedefs.h>

#include "launch.h"
#include "tc_common.cuh"

namespace relattn {
namespace {

using namespace tc;

constexpr int BM = 128, BN = kTcKeyTile;
constexpr int K_STAGES = 2, V_STAGES = 3;
constexpr int NTHREADS = 384;
constexpr float kRescaleThreshold = 8.f;   // log2 units
// Every warp keeps the 168 registers of the launch: the softmax warps fit
// (no spills), and moving registers to them with setmaxnreg measured slower.

constexpr uint32_t TM_O = 0, TM_S = 256;   // O_w at 128 w, S_w at 256 + 128 w

constexpr uint32_t BOX_BYTES = 16384;                // [64 dims x 128 rows], 128-byte rows
constexpr uint32_t TILE_BYTES = 2 * BOX_BYTES;       // 128 dims
constexpr uint32_t SM_Q = 0;                         // Q_0, Q_1
constexpr uint32_t SM_K = SM_Q + 2 * TILE_BYTES;
constexpr uint32_t SM_V = SM_K + K_STAGES * TILE_BYTES;
constexpr uint32_t SM_BAR = SM_V + V_STAGES * TILE_BYTES;
constexpr int B_Q_FULL = 0, B_K_FULL = 1, B_K_EMPTY = B_K_FULL + K_STAGES, B_V_FULL = B_K_EMPTY + K_STAGES,
              B_V_EMPTY = B_V_FULL + V_STAGES, B_S_FULL = B_V_EMPTY + V_STAGES, B_P_FULL = B_S_FULL + 2,
              B_P_HALF = B_P_FULL + 2, B_PV_TAIL = B_P_HALF + 2, B_DRAIN = B_PV_TAIL + 2, B_COUNT = B_DRAIN + 1;
constexpr uint32_t SM_TMEM_SLOT = SM_BAR + B_COUNT * 8;
constexpr uint32_t SM_ABORT = SM_TMEM_SLOT + 8;
constexpr uint32_t SM_TOTAL = SM_ABORT + 8;
constexpr uint32_t SMEM_BYTES = SM_TOTAL + 1024;   // + alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

template <int N>
__device__ __forceinline__ float row_max(const float (&x)[N]) {
  if constexpr (N == 1) {
    return x[0];
  } else if constexpr (N == 2) {
    return fmaxf(x[0], x[1]);
  } else {
    constexpr int M = (N + 2) / 3;
    float t[M];
#pragma unroll
    for (int k = 0; k < M; ++k) {
      if (3 * k + 2 < N) t[k] = fmax3(x[3 * k], x[3 * k + 1], x[3 * k + 2]);
      else if (3 * k + 1 < N) t[k] = fmaxf(x[3 * k], x[3 * k + 1]);
      else t[k] = x[3 * k];
    }
    return row_max(t);
  }
}

__global__ void __launch_bounds__(NTHREADS, 1)
relattn_fwd_tc_main_kernel(const __grid_constant__ KernelArgs a,
                           const __grid_constant__ CUtensorMap map_q,
                           const __grid_constant__ CUtensorMap map_k,
                           const __grid_constant__ CUtensorMap map_v) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sb = smem_addr(smem);
  auto bar = [&](int i) { return sb + SM_BAR + 8u * i; };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM_ABORT);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ------------------------------------------------------------ work item
  const int h0 = 2 * blockIdx.y;                       // heads h0, h0 + 1 (same GQA group)
  const int kv_head = h0 / a.group;
  const int row0 = (a.q_tiles - 1 - blockIdx.x) * BM;  // longest-running tiles first
  const int b = blockIdx.z;
  const int cq = a.cu_q[b], ck = a.cu_k[b];
  const int Lq = a.cu_q[b + 1] - cq, Lk = a.cu_k[b + 1] - ck;
  if (Lq < 0 || Lk < Lq || Lq > a.max_q || Lk > a.max_k) {
    if (tid == 0) atomicOr(a.err, kDevErrSeqlens);
    return;
  }
  const int nrows = min(BM, Lq - row0);
  if (nrows <= 0) return;
  const int off = Lk - Lq;
  const int p0 = off + row0, p_last = p0 + nrows - 1;
  const int j_lo = a.window > 0 ? max(0, p0 - a.window + 1) : 0;
  // 128-key tiles from the diagonal backwards: tile t = keys [p0 - 128 t, p0 - 128 t + 127];
  // the band tiles (some distance < E) are the bias kernel's, the same count it computes
  const int ntiles = (p0 - j_lo + BN - 1) / BN + 1;
  int t_begin = 0;
  if (a.init_from_out) {
    const int lim = a.E + BN - 1;
    t_begin = BN * (ntiles - 1) < lim ? ntiles : min(ntiles, max(0, (lim + BN - 1) / BN));
  }
  const int n_main = ntiles - t_begin;
  if (n_main <= 0) return;   // the band result is final

  // ------------------------------------------------------------ setup
  if (tid == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    for (int i = 0; i < K_STAGES; ++i) {
      mbar_init(bar(B_K_FULL + i), 1);
      mbar_init(bar(B_K_EMPTY + i), 1);
    }
    for (int i = 0; i < V_STAGES; ++i) {
      mbar_init(bar(B_V_FULL + i), 1);
      mbar_init(bar(B_V_EMPTY + i), 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(bar(B_S_FULL + w), 1);
      mbar_init(bar(B_P_FULL + w), 128);
      mbar_init(bar(B_P_HALF + w), 128);
      mbar_init(bar(B_PV_TAIL + w), 1);
    }
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + SM_TMEM_SLOT, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map_q);
    prefetch_tmap(&map_k);
    prefetch_tmap(&map_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + SM_TMEM_SLOT);
  int issued_k = 0, issued_v = 0;   // producer's copies (to drain them if the CTA gives up)
  bool q_issued = false;

  if (warp < 4) {
    if (warp == 0) {
      // ====================================================== TMA producer
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_Q_FULL), 2 * TILE_BYTES);
        for (int w = 0; w < 2; ++w) {
          tma_load_3d(sb + SM_Q + w * TILE_BYTES, &map_q, 0, h0 + w, cq + row0, bar(B_Q_FULL));
          tma_load_3d(sb + SM_Q + w * TILE_BYTES + BOX_BYTES, &map_q, 64, h0 + w, cq + row0, bar(B_Q_FULL));
        }
        q_issued = true;
        for (int i = 0; i < n_main && !*abort_flag; ++i) {
          const int t = t_begin + i;
          const int key = ck + p0 - BN * t;   // may be < 0: the tile reads zeros there
          const int ks = i % K_STAGES, vs = i % V_STAGES;
          if (i >= K_STAGES && !mbar_wait(bar(B_K_EMPTY + ks), ((i / K_STAGES) - 1) & 1, abort_flag, 21)) break;
          if (i != a.test_skip_k_tile) {   // (test hook: a skipped tile is never loaded)
            mbar_arrive_expect_tx(bar(B_K_FULL + ks), TILE_BYTES);
            tma_load_3d(sb + SM_K + ks * TILE_BYTES, &map_k, 0, kv_head, key, bar(B_K_FULL + ks));
            tma_load_3d(sb + SM_K + ks * TILE_BYTES + BOX_BYTES, &map_k, 64, kv_head, key, bar(B_K_FULL + ks));
          }
          issued_k = i + 1;
          if (i >= V_STAGES && !mbar_wait(bar(B_V_EMPTY + vs), ((i / V_STAGES) - 1) & 1, abort_flag, 22)) break;
          mbar_arrive_expect_tx(bar(B_V_FULL + vs), TILE_BYTES);
          tma_load_3d(sb + SM_V + vs * TILE_BYTES, &map_v, 0, kv_head, key, bar(B_V_FULL + vs));
          tma_load_3d(sb + SM_V + vs * TILE_BYTES + BOX_BYTES, &map_v, 64, kv_head, key, bar(B_V_FULL + vs));
          issued_v = i + 1;
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ====================================================== MMA issuer
      // The whole warp runs this (descriptors stay warp-uniform); each MMA and
      // commit is issued by one elected lane.
      {
        const uint32_t id_s = idesc_bf16_f32(BM, BN, 0, 0);     // S: Q (smem, K-major) x K (smem, K-major)
        const uint32_t id_o = idesc_bf16_f32(BM, 128, 0, 1);    // O: P (tmem) x V (smem, MN-major)
        // descriptor bases: +2 per 32 bytes of a 128-byte row, +1024 per 16 KB
        // box, +128 per 16 V rows, +2048 per 32 KB tile
        const uint64_t qd0 = smem_desc_sw128(sb + SM_Q, 16, 1024);
        const uint64_t kd0 = smem_desc_sw128(sb + SM_K, 16, 1024);
        const uint64_t vd0 = smem_desc_sw128(sb + SM_V, BOX_BYTES, 1024);
        bool ok = mbar_wait_warp(bar(B_Q_FULL), 0, abort_flag, 23);
        auto issue_s = [&](int w, int i) -> bool {   // S_w of main tile i
          const int ks = i % K_STAGES;
          if (w == 0 && !mbar_wait_warp(bar(B_K_FULL + ks), (i / K_STAGES) & 1, abort_flag, 24)) return false;
          const uint64_t qd = qd0 + (uint64_t)(w * (TILE_BYTES >> 4));
          const uint64_t kd = kd0 + (uint64_t)(ks * (TILE_BYTES >> 4));
          const uint32_t d = tmem + TM_S + 128u * (uint32_t)w;
          mma_ss_e<0>(d, qd + 0, kd + 0, id_s);
          mma_ss_e<1>(d, qd + 2, kd + 2, id_s);
          mma_ss_e<1>(d, qd + 4, kd + 4, id_s);
          mma_ss_e<1>(d, qd + 6, kd + 6, id_s);
          mma_ss_e<1>(d, qd + 1024, kd + 1024, id_s);
          mma_ss_e<1>(d, qd + 1026, kd + 1026, id_s);
          mma_ss_e<1>(d, qd + 1028, kd + 1028, id_s);
          mma_ss_e<1>(d, qd + 1030, kd + 1030, id_s);
          mma_commit_e(bar(B_S_FULL + w));
          return true;
        };
        // O_w += P_w V of main tile i, keys 0..63 once the softmax has written
        // that half of P, keys 64..127 once it has written all of it
        auto issue_pv = [&](int w, int i) -> bool {
          const int vs = i % V_STAGES;
          if (w == 0 && !mbar_wait_warp(bar(B_V_FULL + vs), (i / V_STAGES) & 1, abort_flag, 25)) return false;
          if (!mbar_wait_warp(bar(B_P_HALF + w), i & 1, abort_flag, 30)) return false;
          tc_fence_after();
          const uint64_t vd = vd0 + (uint64_t)(vs * (TILE_BYTES >> 4));
          const uint32_t o = tmem + TM_O + 128u * (uint32_t)w, pa = tmem + TM_S + 128u * (uint32_t)w;
          if (i > 0 || a.init_from_out) mma_ts_e<1>(o, pa + 0, vd + 0, id_o);
          else mma_ts_e<0>(o, pa + 0, vd + 0, id_o);
          mma_ts_e<1>(o, pa + 8, vd + 128, id_o);
          mma_ts_e<1>(o, pa + 16, vd + 256, id_o);
          mma_ts_e<1>(o, pa + 24, vd + 384, id_o);
          if (!mbar_wait_warp(bar(B_P_FULL + w), i & 1, abort_flag, 26)) return false;
          tc_fence_after();
          mma_ts_e<1>(o, pa + 32, vd + 512, id_o);
          mma_ts_e<1>(o, pa + 40, vd + 640, id_o);
          mma_ts_e<1>(o, pa + 48, vd + 768, id_o);
          mma_ts_e<1>(o, pa + 56, vd + 896, id_o);
          if (i == n_main - 1) mma_commit_e(bar(B_PV_TAIL + w));
          return true;
        };
        if (ok) ok = issue_s(0, 0);
        if (ok) ok = issue_s(1, 0);
        // S_w(i+1) goes into the buffer whose P_w(i) PV_w(i) has just been
        // issued to read: the tensor core runs them in order
        for (int i = 0; i < n_main && ok; ++i) {
          for (int w = 0; w < 2 && ok; ++w) {
            if (!(ok = issue_pv(w, i))) break;
            if (i + 1 < n_main) ok = issue_s(w, i + 1);
          }
        }
        // drain: every MMA issued above has finished before TMEM is released
        mma_commit_e(bar(B_DRAIN));
        volatile int keep_waiting = 0;
        mbar_wait(bar(B_DRAIN), 0, &keep_waiting, 27, 400000000ll);
      }
      __syncwarp();
    }
  } else {
    // ======================================================== softmax
    const int w = (warp - 4) >> 2;               // head h0 + w
    const int wq = warp & 3;                     // lane quarter (TMEM lanes 32 wq ..)
    const int a_row = 32 * wq + lane;            // row == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    const int h = h0 + w;
    const int t_row = min(row0 + a_row, Lq - 1);
    const int pos = p0 + a_row;                  // padding rows continue the pattern
    const float sc = log_scale(min(pos, p_last), a.inv_ln_base);
    const float cqk = a.alpha_log2e * sc;        // > 0 (checked on the host)
    const bool releaser = (w == 1) && (wq == 0) && (lane == 0);   // frees K / V stages
    const uint32_t obuf = tmem + lane_base + TM_O + 128u * (uint32_t)w;
    const uint32_t sbuf = tmem + lane_base + TM_S + 128u * (uint32_t)w;
    const size_t qrow = (size_t)(cq + t_row) * a.Hq + h;
    auto warp_wait = [&](uint32_t br, uint32_t parity, int site) -> bool {
      const bool r = mbar_wait(br, parity, abort_flag, site);
      return __all_sync(0xffffffffu, r);
    };

    float m_ref = -INFINITY, l = 0.f;
    if (a.init_from_out) {
      // the band's state: m = lse log2(e), l = 1, O = out (normalised)
      const float lse0 = a.lse[(size_t)h * a.total_q + cq + t_row];
      if (lse0 != -INFINITY) {
        m_ref = lse0 * kLog2e;
        l = 1.f;
      }
      const uint4 *src = reinterpret_cast<const uint4 *>(a.out + qrow * kHeadDim);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = src[4 * c + i];
          const uint32_t pr[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            r[8 * i + 2 * k] = __float_as_uint(__uint_as_float(pr[k] << 16));
            r[8 * i + 2 * k + 1] = __float_as_uint(__uint_as_float(pr[k] & 0xffff0000u));
          }
        }
        __syncwarp();
        tmem_st32(obuf + 32u * c, r);
      }
      tmem_wait_st();
    }

    bool ok = true;
    for (int i = 0; i < n_main; ++i) {
      const int t = t_begin + i;
      if (!(ok = warp_wait(bar(B_S_FULL + w), i & 1, 28))) break;
      if (releaser) {
        // S_1(i) landed: K(i) is read by both heads; S_1(i) was issued after
        // PV_1(i-1), so V(i-1) is free too
        mbar_arrive(bar(B_K_EMPTY + i % K_STAGES));
        if (i > 0) mbar_arrive(bar(B_V_EMPTY + (i - 1) % V_STAGES));
      }
      tc_fence_after();
      float x[128];   // raw scores; the scale is applied inside the exponent
      __syncwarp();
      tmem_ld32f<0>(sbuf + 0u, x);
      tmem_ld32f<32>(sbuf + 32u, x);
      tmem_ld32f<64>(sbuf + 64u, x);
      tmem_ld32f<96>(sbuf + 96u, x);
      tmem_wait_ld_f<0>(x);
      reg_dep_f<32>(x);
      reg_dep_f<64>(x);
      reg_dep_f<96>(x);
      const int j0 = p0 - BN * t;
      const bool need_mask = (j0 + BN - 1 > p0) || (a.window > 0 && j0 < p_last - a.window + 1) || (j0 < 0);
      if (need_mask) {
        // visible keys of this row are one range [kmin, kmax] of the tile
        const int kmax = pos - j0;
        const int kmin = max(-j0, a.window > 0 ? pos - a.window + 1 - j0 : 0);
#pragma unroll
        for (int k = 0; k < 128; ++k) x[k] = (k >= kmin && k <= kmax) ? x[k] : -INFINITY;
      }
      // P (bf16 pairs) of keys 32c .. 32c + 31 over S_w columns [16c, 16c + 16)
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      auto p_chunk = [&](int c, float mu) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float y0, y1;
          ffma2(y0, y1, x[32 * c + 2 * k], x[32 * c + 2 * k + 1], cqk, cqk, -mu, -mu);
          const float e0 = fast_exp2(y0), e1 = fast_exp2(y1);
          ffma2(acc[2 * (k & 1)], acc[2 * (k & 1) + 1], e0, e1, 1.f, 1.f, acc[2 * (k & 1)], acc[2 * (k & 1) + 1]);
          pk[k] = pack_bf16x2(e0, e1);
        }
        __syncwarp();
        tmem_st16(sbuf + 16u * (uint32_t)c, pk);
      };
      // Where every row of the warp has a running max, the first half of P is
      // computed against it before the tile's own max is known: that max only
      // decides whether the running max moves (a rare rescale), and a warp in
      // which some row's does recomputes the half.  The values are the same as
      // computing the max first.
      const bool spec = __all_sync(0xffffffffu, m_ref != -INFINITY);
      if (spec) {
        p_chunk(0, m_ref);
        p_chunk(1, m_ref);
      }
      const float mx = row_max(x) * cqk;
      float corr = 1.f;
      bool rescale_o = false, moved = false;
      if (mx > m_ref + kRescaleThreshold || (m_ref == -INFINITY && mx != -INFINITY)) {
        const float m_new = fmaxf(m_ref, mx);
        corr = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - m_new);
        rescale_o = (m_ref != -INFINITY) && (i > 0 || a.init_from_out);
        l *= corr;
        m_ref = m_new;
        moved = true;
      }
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      if (!spec || __any_sync(0xffffffffu, moved)) {
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = 0.f;
        p_chunk(0, m_use);
        p_chunk(1, m_use);
      }
      // O_w is touched only when a row of this warp needs a rescale; PV_w(i-1)
      // has finished (S_w(i) was issued after it).  TMEM loads / stores are
      // warp-collective: the whole warp rescales (rows that need not: by 1).
      // It happens before the first half of P is handed over: PV_w(i) starts then.
      if (__any_sync(0xffffffffu, rescale_o)) {
        const float cf = rescale_o ? corr : 1.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          __syncwarp();
          tmem_ld32(obuf + 32u * c, r);
          tmem_wait_ld(r);
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * cf);
          __syncwarp();
          tmem_st32(obuf + 32u * c, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_P_HALF + w));
      p_chunk(2, m_use);
      p_chunk(3, m_use);
      l += (acc[0] + acc[1]) + (acc[2] + acc[3]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_P_FULL + w));
    }
    // ---- epilogue
    if (ok) ok = warp_wait(bar(B_PV_TAIL + w), 0, 29);
    if (ok) {
      tc_fence_after();
      const bool valid = a_row < nrows;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float row_lse = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(obuf + 32u * c, r);
        tmem_wait_ld(r);
        if (valid) {
          __nv_bfloat16 *dst = a.out + qrow * kHeadDim + 32 * c;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(r[8 * k + 0]) * inv, __uint_as_float(r[8 * k + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(r[8 * k + 2]) * inv, __uint_as_float(r[8 * k + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(r[8 * k + 4]) * inv, __uint_as_float(r[8 * k + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(r[8 * k + 6]) * inv, __uint_as_float(r[8 * k + 7]) * inv);
            *reinterpret_cast<uint4 *>(dst + 8 * k) = v;
          }
        }
      }
      if (valid) a.lse[(size_t)h * a.total_q + cq + t_row] = row_lse;
    }
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) record_timeout(a.err, *abort_flag);
  if (warp == 0 && lane == 0 && *abort_flag) {
    // the CTA gave up: let the producer's own copies land before shared memory
    // goes away (bounded waits, not cut short by the abort)
    volatile int keep_waiting = 0;
    if (q_issued) mbar_wait(bar(B_Q_FULL), 0, &keep_waiting, 2, 400000000ll);
    for (int i = max(0, issued_k - K_STAGES); i < issued_k; ++i)
      if (i != a.test_skip_k_tile)
        mbar_wait(bar(B_K_FULL + i % K_STAGES), (i / K_STAGES) & 1, &keep_waiting, 2, 400000000ll);
    for (int i = max(0, issued_v - V_STAGES); i < issued_v; ++i)
      mbar_wait(bar(B_V_FULL + i % V_STAGES), (i / V_STAGES) & 1, &keep_waiting, 2, 400000000ll);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// [rows, heads, 128] bf16 -> box of 64 dims x 1 head x 128 rows, 128-byte swizzle
bool encode_rows(CUtensorMap *m, const void *base, int heads, int rows) {
  auto fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {256, (cuuint64_t)heads * 256};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)BN};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_main_supported(const KernelArgs &a, int total_q, int total_k) {
  // two heads of one GQA group per CTA; a positive score scale; 128-row TMA
  // boxes inside the tensors
  return encoder() && a.group % 2 == 0 && a.alpha_log2e > 0.f && total_q >= BM && total_k >= BN;
}

cudaError_t launch_prefill_tc_main(const KernelArgs &a, int total_k, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (!encode_rows(&mq, a.q, a.Hq, a.total_q)) return cudaErrorInvalidValue;
  if (!encode_rows(&mk, a.k, a.Hkv, total_k)) return cudaErrorInvalidValue;
  if (!encode_rows(&mv, a.v, a.Hkv, total_k)) return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[kMaxDevicesAttr];
  cudaError_t e = set_max_smem_once(reinterpret_cast<const void *>(relattn_fwd_tc_main_kernel),
                                    (int)SMEM_BYTES, attr_set);
  if (e != cudaSuccess) return e;
  relattn_fwd_tc_main_kernel<<<dim3(a.q_tiles, a.Hq / 2, a.batch), NTHREADS, SMEM_BYTES, stream>>>(
      a, mq, mk, mv);
  return cudaGetLastError();
}

}  // namespace relattn
