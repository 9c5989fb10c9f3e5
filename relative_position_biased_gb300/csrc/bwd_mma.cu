// bwd_mma.cu -- backward pass of relative attention on warp-level bf16 MMAs
// (mma.sync m16n8k16), P frozen.
//
// Page "SGLang and Miles Add Day-0 Support for Inkling", section "Customized
// Efficient Kernels for Train-Inference Consistency", paragraph "Relative
// attention": the training side differentiates through the attention scores
// and through r while P stays fixed.  With
//     l(i,j) = s_i (alpha q_i.k_j + [0 <= i-j < E] r_i.P[:, i-j]),
//     p(i,j) = exp(l(i,j) - lse_i),   out_i = sum_j p(i,j) v_j,
// the gradients of sum(dout * out) are
//     D_i = dout_i . out_i,            dl(i,j) = p(i,j) (dout_i . v_j - D_i),
//     dq_i = s_i alpha sum_j dl(i,j) k_j,      dk_j = sum_i s_i alpha dl(i,j) q_i,
//     dv_j = sum_i p(i,j) dout_i,              dr_i = s_i sum_j dl(i,j) P[:, i-j]
// (dk, dv also summed over the query heads of a GQA group).
//
// Up to five launches, no atomics:
//   0. relattn_bwd_rel_kernel (with a bias, before the tcgen05 dk / dv): R = r . P
//      for every row, head and distance below E (fp32, in the workspace), the
//      windows that kernel loads by TMA;
//   1. relattn_bwd_dot_kernel: D = rowsum(dout * out) (fp32, [Hq, Tq]).
//   2. dq over the keys every row of a 128-row tile sees outside the bias band
//      (all keys without a bias), on tcgen05 (bwd_tc.cu) when the shapes allow;
//      with a bias its fp32 result goes to the workspace.
//   3. relattn_bwd_dq_kernel for the remaining keys (all keys without tcgen05),
//      adding 2.'s part; it writes dq and dr: a CTA takes 64 query rows of one
//      head and walks the key tiles they see, recomputing S (with the bias
//      band, as the forward does) and P from the saved lse, then dP = dout V^T,
//      dS = P (dP - D); dq += dS K in registers.  Inside the bias band dS is
//      sheared into a per-group [row, distance] window in shared memory and
//      dr += window . P_slice^T on the tensor cores.
//   4. dk / dv, key-major: on tcgen05 (bwd_tc.cu) when the shapes allow, else
//      relattn_bwd_dkdv_kernel here: a CTA takes 64 keys of one kv head and
//      walks the (query head, query tile) pairs that see them; per pair it
//      computes the bias window R = r . P_slice once into shared memory, then
//      per warp (16 keys) S^T, P^T, dP^T = V dout^T, dS^T, and
//      dv += P^T dout, dk += dS^T q in registers.
// All recompute S and P (the forward's P is not stored).  Here K / V (kernel 3)
// and q / dout / r / lse / D (kernel 4) stream through 2-stage cp.async rings.
#include "launch.h"

namespace relattn {
namespace {

constexpr int BT = 64;              // query rows and keys per tile
constexpr int NWB = 8;              // warps per CTA: 4 groups of 16 rows (or keys) x 2 halves
constexpr int NTB = NWB * 32;
constexpr int NGRP = 4;             // 16-row (16-key) groups per 64-row (64-key) tile
constexpr int BSTAGES = 2;
constexpr int RWQ = 88;             // dq kernel: R / dS window columns per warp
constexpr int DSW = 104;            // bf16 row stride of the dS window (96 used)
constexpr int PWQ = 152;            // dq kernel: P slice columns per stage
constexpr int PWK = 136;            // dkdv kernel: P slice / R window columns
// bf16 row stride of a P slice: PW + pad with (PW + pad) / 8 odd, so the 8
// rows of an ldmatrix 8x8 load fall in 8 different 16-byte bank groups
__host__ __device__ constexpr int p_stride(int pw) { return ((pw / 8 + 1) | 1) * 8; }
constexpr int RSK = 163;            // dkdv kernel: fp32 row stride of R (conflict-free gather)

__device__ __forceinline__ int floor8(int x) { return x & ~7; }

__device__ __forceinline__ void ldsm_x4_n(uint32_t addr, uint32_t (&r)[4]) {
  ldsm_x4(addr, r[0], r[1], r[2], r[3]);
}

// swizzled 256-byte row: 16-byte chunk c of row `row`
__device__ __forceinline__ uint32_t swz(int row, int c) { return row * 256 + ((c ^ (row & 7)) << 4); }

// P columns [cb, cb + PW) of all rd_pad channels into a [rd_pad][p_stride(PW)]
// bf16 slice; columns outside [0, E) and channels past rd read as zero.
template <int PW>
__device__ __forceinline__ void load_p_slice(const BwdArgs &a, uint32_t base, int cb, int tid) {
  constexpr int PS = p_stride(PW), cpr = PW / 8;
  for (int idx = tid; idx < a.rd_pad * cpr; idx += NTB) {
    const int c = idx / cpr, x = idx - c * cpr, col = cb + x * 8;
    const uint32_t dst = base + (c * PS + x * 8) * 2;
    const bool in_row = c < a.rd;
    const bool whole = col >= 0 && col + 8 <= a.E;
    const bool none = !in_row || col + 8 <= 0 || col >= a.E;
    if (a.p_vec_ok && (whole || none)) {
      const bool ok = in_row && whole;
      cp_async16(dst, a.P + (ok ? (size_t)c * a.E + col : 0), ok);
    } else {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c0 = col + 2 * e, c1 = c0 + 1;
        const unsigned short lo = (in_row && c0 >= 0 && c0 < a.E) ? __bfloat16_as_ushort(a.P[(size_t)c * a.E + c0]) : 0;
        const unsigned short hi = (in_row && c1 >= 0 && c1 < a.E) ? __bfloat16_as_ushort(a.P[(size_t)c * a.E + c1]) : 0;
        w[e] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      st_shared_v4(dst, w[0], w[1], w[2], w[3]);
    }
  }
}

// ------------------------------------------------------------------ D = rowsum(dout * out)

__global__ void __launch_bounds__(256) relattn_bwd_dot_kernel(const BwdArgs a) {
  // a half-warp per (t, h) row, 8 dims a lane
  const long rows = (long)a.total_q * a.Hq;
  const int hl = threadIdx.x & 15;
  const unsigned hmask = 0xffffu << (threadIdx.x & 16);
  for (long row = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 4; row < rows;
       row += ((long)gridDim.x * blockDim.x) >> 4) {
    const uint4 o = *reinterpret_cast<const uint4 *>(a.out + row * kHeadDim + 8 * hl);
    const uint4 d = *reinterpret_cast<const uint4 *>(a.dout + row * kHeadDim + 8 * hl);
    const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, dw[4] = {d.x, d.y, d.z, d.w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(ow[i] << 16), __uint_as_float(dw[i] << 16), acc);
      acc = fmaf(__uint_as_float(ow[i] & 0xffff0000u), __uint_as_float(dw[i] & 0xffff0000u), acc);
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(hmask, acc, off);
    if (hl == 0) {
      const long t = row / a.Hq, h = row - t * a.Hq;
      a.Dsum[h * a.total_q + t] = acc;
    }
  }
}

// ------------------------------------------------------------------ R = r . P for every row

// Rall[(t, h)][d] = r_{t,h} . P[:, d] for d < E (fp32 accumulation of bf16
// products, as the forward's r.P): a [Tq*Hq, r_dim] x [r_dim, E] product. A
// CTA keeps one 128-row r tile in shared memory and walks E in 128-distance
// chunks, 8 warps of 16 rows.  The tcgen05 dk / dv loads its bias windows
// from it instead of recomputing them per tile.
constexpr int RPT = 128;
__global__ void __launch_bounds__(256) relattn_bwd_rel_kernel(const BwdArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, qq = lane & 3;
  const long rows = (long)a.total_q * a.Hq;
  const long row0 = (long)blockIdx.x * RPT;
  const int rs = (a.rd_pad + 8) * 2;                  // bytes per r-tile row (odd 16-byte units)
  const uint32_t pbase = sbase + RPT * rs;
  const int rcs = a.rd_pad / 8;
  for (int idx = tid; idx < RPT * rcs; idx += 256) {   // the r tile, once for all of E
    const int r = idx / rcs, c = idx - r * rcs;
    const bool ok = row0 + r < rows && c * 8 < a.rd;
    cp_async16(sbase + r * rs + c * 16, a.r + (ok ? (row0 + r) * a.rd + c * 8 : 0), ok);
  }
  constexpr int PS = p_stride(RPT), cpr = RPT / 8;
  for (int c0 = 0; c0 < a.E; c0 += RPT) {             // 128-distance chunks of E
    if (c0 > 0) __syncthreads();                       // the previous chunk's P slice is read
    for (int idx = tid; idx < a.rd_pad * cpr; idx += 256) {
      const int c = idx / cpr, x = idx - c * cpr, col = c0 + x * 8;
      const uint32_t dst = pbase + (c * PS + x * 8) * 2;
      const bool in_row = c < a.rd;
      if (a.p_vec_ok && in_row && col + 8 <= a.E) {
        cp_async16(dst, a.P + (size_t)c * a.E + col, true);
      } else {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d0 = col + 2 * e, d1 = d0 + 1;
          const unsigned short lo = (in_row && d0 < a.E) ? __bfloat16_as_ushort(a.P[(size_t)c * a.E + d0]) : 0;
          const unsigned short hi = (in_row && d1 < a.E) ? __bfloat16_as_ushort(a.P[(size_t)c * a.E + d1]) : 0;
          w[e] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        st_shared_v4(dst, w[0], w[1], w[2], w[3]);
      }
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    float acc[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    for (int kk = 0; kk < a.rd_pad / 16; ++kk) {
      uint32_t ra[4];
      ldsm_x4_n(sbase + (warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3)) * rs +
                    (kk * 16 + ((lane >> 4) << 3)) * 2, ra);
      const int prow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(pbase + (prow * PS + np * 16 + ((lane >> 4) << 3)) * 2, b0, b1, b2, b3);
        mma_bf16_16816(acc[2 * np], ra[0], ra[1], ra[2], ra[3], b0, b1);
        mma_bf16_16816(acc[2 * np + 1], ra[0], ra[1], ra[2], ra[3], b2, b3);
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const long row = row0 + warp * 16 + gq + 8 * r;
      if (row >= rows) continue;
      float *dst = a.Rall + row * a.e_pad;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const int col = c0 + n * 8 + 2 * qq;
        // distances E .. e_pad - 1 (the row's padding) are written as zeros
        if (col + 1 < a.E) {
          *reinterpret_cast<float2 *>(dst + col) = make_float2(acc[n][2 * r], acc[n][2 * r + 1]);
        } else if (col < a.e_pad) {
          dst[col] = col < a.E ? acc[n][2 * r] : 0.f;
          if (col + 1 < a.e_pad) dst[col + 1] = 0.f;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ dq / dr (query-major)

struct DqLayout {
  static constexpr int q = 0;                              // Q tile [64][128] swizzled
  static constexpr int dout = q + BT * 256;                // dout tile
  static constexpr int win = dout + BT * 256;              // per-group R (fp32 16 x 88) / dS windows
  static constexpr int win_bytes = 16 * RWQ * 4;
  static constexpr int kv = win + NGRP * win_bytes;        // K, V ring
  static constexpr int kv_stage = BT * 256;
  static constexpr int p = kv + 2 * BSTAGES * kv_stage;    // P slice ring
  __host__ __device__ static int p_stage(int rd_pad) { return rd_pad * p_stride(PWQ) * 2; }
  __host__ __device__ static int r(int rd_pad) { return p + BSTAGES * p_stage(rd_pad); }
  __host__ __device__ static int r_stride(int rd_pad) { return (rd_pad + 8) * 2; }
  // R windows loaded from the precomputed R (a ring beside K / V)
  static constexpr int rw_stage = NGRP * win_bytes;
  __host__ __device__ static int rw(int rd_pad) { return r(rd_pad) + BT * r_stride(rd_pad); }
  __host__ __device__ static int total(int rd_pad) { return rw(rd_pad) + BSTAGES * rw_stage; }
};
static_assert(DqLayout::kv % 16 == 0 && DqLayout::win_bytes % 16 == 0, "16-byte copies");

// Warp (rw, kh) takes query rows 16 rw .. 16 rw + 15 and keys 32 kh .. 32 kh + 31
// of every key tile; the two warps of a row group share that group's R / dS
// window and sum their partial dq / dr at the end.
__global__ void __launch_bounds__(NTB, 1) relattn_bwd_dq_kernel(const __grid_constant__ BwdArgs a) {
  using L = DqLayout;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, qq = lane & 3;
  const int rw = warp & (NGRP - 1), kh = warp / NGRP;

  const int q_tile = a.q_tiles - 1 - blockIdx.x;   // longest first
  const int h = blockIdx.y, b = blockIdx.z;
  const int cq = a.cu_q[b], ck = a.cu_k[b];
  const int Lq = a.cu_q[b + 1] - cq, Lk = a.cu_k[b + 1] - ck;
  if (Lq < 0 || Lk < Lq || Lq > a.max_q || Lk > a.max_k) {
    if (tid == 0) atomicOr(a.err, kDevErrSeqlens);
    return;
  }
  const int row0 = q_tile * BT;
  const int nrows = min(BT, Lq - row0);
  if (nrows <= 0) return;
  const int off = Lk - Lq, g = h / a.group;
  const int p_min = off + row0, p_max = off + row0 + nrows - 1;
  const int j_lo = a.window > 0 ? max(0, p_min - a.window + 1) : 0;
  int kbeg = j_lo & ~(BT - 1);
  if (a.dq_split) {
    // keys every row of the enclosing 128-row tile sees outside the band are
    // the tcgen05 dq's (relattn_bwd_dq_tc_kernel, same bound)
    const int p0 = off + (row0 & ~127);
    kbeg = max(kbeg, p0 - a.E + 1 > 0 ? (p0 - a.E + 1) & ~63 : 0);
  }
  const int kend = p_max + 1;
  const int ntiles = (kend - kbeg + BT - 1) / BT;
  auto tile_j0 = [&](int it) { return kbeg + (ntiles - 1 - it) * BT; };   // diagonal first
  const bool has_bias = a.rd > 0 && a.E > 0;
  const bool use_rall = has_bias && a.rall_ok;
  auto is_band = [&](int j0) { return has_bias && (p_min - (j0 + BT - 1) < a.E); };

  auto issue_tile = [&](int it) {
    const int j0 = tile_j0(it), st = it % BSTAGES;
    for (int idx = tid; idx < BT * 16; idx += NTB) {
      const int row = idx >> 4, c = idx & 15, j = j0 + row;
      const bool ok = j < Lk;
      const size_t gi = ((size_t)(ck + (ok ? j : 0)) * a.Hkv + g) * kHeadDim + c * 8;
      cp_async16(sbase + L::kv + st * L::kv_stage + swz(row, c), a.k + gi, ok);
      cp_async16(sbase + L::kv + (BSTAGES + st) * L::kv_stage + swz(row, c), a.v + gi, ok);
    }
    if (is_band(j0)) {
      load_p_slice<PWQ>(a, sbase + L::p + st * L::p_stage(a.rd_pad), floor8(p_min - j0 - BT), tid);
      if (use_rall) {
        // each group's R window, R[row][cbw_g .. cbw_g + 88), in 16-byte pieces;
        // cbw_g is a multiple of 8, so a piece is inside a row's [0, e_pad)
        // (the padding past E holds zeros) or wholly outside it (zero-filled)
        constexpr int PR = RWQ / 4;                        // pieces per row
        for (int idx = tid; idx < NGRP * 16 * PR; idx += NTB) {
          const int gg = idx / (16 * PR), rem = idx - gg * 16 * PR, rr = rem / PR, k = rem - rr * PR;
          const int cbw_g = floor8(off + row0 + min(16 * gg, nrows - 1) - j0 - BT);
          const int d = cbw_g + 4 * k;
          const bool ok = d >= 0 && d < a.e_pad;
          const float *src = a.Rall + ((size_t)(cq + row0 + min(16 * gg + rr, nrows - 1)) * a.Hq + h) * a.e_pad;
          cp_async16(sbase + L::rw(a.rd_pad) + st * L::rw_stage + gg * L::win_bytes + (rr * RWQ + 4 * k) * 4,
                     ok ? src + d : a.Rall, ok);
        }
      }
    }
  };

  // Q, dout, r rows of the tile (rows past the end are clamped to the last one)
  for (int idx = tid; idx < BT * 16; idx += NTB) {
    const int row = idx >> 4, c = idx & 15;
    const size_t gi = ((size_t)(cq + row0 + min(row, nrows - 1)) * a.Hq + h) * kHeadDim + c * 8;
    cp_async16(sbase + L::q + swz(row, c), a.q + gi, true);
    cp_async16(sbase + L::dout + swz(row, c), a.dout + gi, true);
  }
  if (has_bias && !use_rall) {
    const int rcs = a.rd_pad / 8;
    for (int idx = tid; idx < BT * rcs; idx += NTB) {
      const int row = idx / rcs, c = idx - row * rcs;
      const __nv_bfloat16 *src = a.r + ((size_t)(cq + row0 + min(row, nrows - 1)) * a.Hq + h) * a.rd;
      cp_async16(sbase + L::r(a.rd_pad) + row * L::r_stride(a.rd_pad) + c * 16,
                 src + (c * 8 < a.rd ? c * 8 : 0), c * 8 < a.rd);
    }
  }
#pragma unroll
  for (int s = 0; s < BSTAGES - 1; ++s) {
    if (s < ntiles) issue_tile(s);
    cp_async_commit();
  }

  // per-row constants: the two rows gq, gq + 8 of this group
  float cqk[2], cbias[2], lse2[2], Dr[2], srow[2];
  int pos[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int rl = min(rw * 16 + gq + 8 * r, nrows - 1);
    pos[r] = off + row0 + rl;
    srow[r] = log_scale(pos[r], a.inv_ln_base);
    cqk[r] = a.alpha_log2e * srow[r];
    cbias[r] = kLog2e * srow[r];
    lse2[r] = a.lse[(size_t)h * a.total_q + cq + row0 + rl] * kLog2e;
    Dr[r] = a.Dsum[(size_t)h * a.total_q + cq + row0 + rl];
  }
  const int p_w0 = off + row0 + min(rw * 16, nrows - 1);

  float dq[16][4], dr[8][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) dq[n][0] = dq[n][1] = dq[n][2] = dq[n][3] = 0.f;
#pragma unroll
  for (int n = 0; n < 8; ++n) dr[n][0] = dr[n][1] = dr[n][2] = dr[n][3] = 0.f;
  float *win = reinterpret_cast<float *>(smem + L::win + rw * L::win_bytes);
  const uint32_t win_s = sbase + L::win + rw * L::win_bytes;
  const int arow = rw * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);   // A-operand ldmatrix row
  const int kb0 = 32 * kh;                                            // this warp's first key
  uint32_t qa[8][4], da[8][4];   // the group's Q / dout rows as A fragments (loaded once)

  for (int it = 0; it < ntiles; ++it) {
    cp_async_wait<BSTAGES - 2>();
    __syncthreads();
    if (it == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        ldsm_x4_n(sbase + L::q + swz(arow, 2 * kk + (lane >> 4)), qa[kk]);
        ldsm_x4_n(sbase + L::dout + swz(arow, 2 * kk + (lane >> 4)), da[kk]);
      }
    }
    if (it + BSTAGES - 1 < ntiles) issue_tile(it + BSTAGES - 1);
    cp_async_commit();
    const int st = it % BSTAGES, j0 = tile_j0(it);
    const uint32_t kb = sbase + L::kv + st * L::kv_stage;
    const uint32_t vb = sbase + L::kv + (BSTAGES + st) * L::kv_stage;
    const bool band = is_band(j0);
    const int cb = floor8(p_min - j0 - BT), cbw = floor8(p_w0 - j0 - BT), coloff = cbw - cb;
    const uint32_t pb = sbase + L::p + st * L::p_stage(a.rd_pad);

    if (band && !use_rall) {
      // the group's R window = r_rows . P[:, cbw .. cbw + 88) (fp32); warp kh
      // computes n8 tiles [6 kh, 6 kh + 6) of the 11.  (Computing it here from
      // shared-memory r and P beats gathering it from the precomputed R: that
      // gather is a DRAM round trip in the inner loop with nothing to hide it.)
      const uint32_t rb = sbase + L::r(a.rd_pad);
      const int rstride = L::r_stride(a.rd_pad);
      constexpr int NH = 6;
      const int nt0 = NH * kh;
      float racc[NH][4];
#pragma unroll
      for (int n = 0; n < NH; ++n) racc[n][0] = racc[n][1] = racc[n][2] = racc[n][3] = 0.f;
      for (int kk = 0; kk < a.rd_pad / 16; ++kk) {
        uint32_t ra[4];
        ldsm_x4_n(rb + arow * rstride + (kk * 16 + ((lane >> 4) << 3)) * 2, ra);
        const int prow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int np = 0; np < NH / 2; ++np) {
          const int nt = nt0 + 2 * np;
          if (nt + 1 < RWQ / 8) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(pb + (prow * p_stride(PWQ) + coloff + nt * 8 + ((lane >> 4) << 3)) * 2, b0, b1, b2, b3);
            mma_bf16_16816(racc[2 * np], ra[0], ra[1], ra[2], ra[3], b0, b1);
            mma_bf16_16816(racc[2 * np + 1], ra[0], ra[1], ra[2], ra[3], b2, b3);
          } else if (nt < RWQ / 8) {
            uint32_t b0, b1;
            ldsm_x2_t(pb + (prow * p_stride(PWQ) + coloff + nt * 8) * 2, b0, b1);
            mma_bf16_16816(racc[2 * np], ra[0], ra[1], ra[2], ra[3], b0, b1);
          }
        }
      }
#pragma unroll
      for (int n = 0; n < NH; ++n) {
        const int nt = nt0 + n;
        if (nt < RWQ / 8) {
          *reinterpret_cast<float2 *>(&win[gq * RWQ + nt * 8 + 2 * qq]) = make_float2(racc[n][0], racc[n][1]);
          *reinterpret_cast<float2 *>(&win[(gq + 8) * RWQ + nt * 8 + 2 * qq]) = make_float2(racc[n][2], racc[n][3]);
        }
      }
    }

    // ---- S = Q K^T and dP = dout V^T (16 rows x this warp's 32 keys)
    float s[4][4], dp[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
      dp[n][0] = dp[n][1] = dp[n][2] = dp[n][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int row = kb0 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = 2 * kk + ((lane >> 3) & 1);
        uint32_t kf[4], vf[4];
        ldsm_x4_n(kb + swz(row, c), kf);
        ldsm_x4_n(vb + swz(row, c), vf);
        mma_bf16_16816(s[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], kf[0], kf[1]);
        mma_bf16_16816(s[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], kf[2], kf[3]);
        mma_bf16_16816(dp[2 * np], da[kk][0], da[kk][1], da[kk][2], da[kk][3], vf[0], vf[1]);
        mma_bf16_16816(dp[2 * np + 1], da[kk][0], da[kk][1], da[kk][2], da[kk][3], vf[2], vf[3]);
      }
    }

    // ---- logits in log2 units: s_i log2e (alpha q.k + bias)
    if (band) {
      if (!use_rall) __syncthreads();    // the group's window is complete
      const float *rwin = use_rall ? reinterpret_cast<const float *>(smem + L::rw(a.rd_pad) + st * L::rw_stage +
                                                                     rw * L::win_bytes)
                                   : win;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float *rrow = rwin + (gq + 8 * r) * RWQ + (pos[r] - j0 - cbw);
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int bcol = kb0 + n * 8 + 2 * qq + e;
            s[n][2 * r + e] = fmaf(s[n][2 * r + e], cqk[r], rrow[-bcol] * cbias[r]);
          }
      }
    } else {
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        s[n][0] *= cqk[0];
        s[n][1] *= cqk[0];
        s[n][2] *= cqk[1];
        s[n][3] *= cqk[1];
      }
    }

    // ---- P = exp2(x - lse2) on the visible keys, dS = P (dP - D)
    const bool need_mask = (j0 + BT - 1 > p_min) ||
                           (a.window > 0 && j0 < p_max - a.window + 1) || (j0 + BT > Lk);
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float x = s[n][2 * r + e];
          if (need_mask) {
            const int j = j0 + kb0 + n * 8 + 2 * qq + e;
            const bool vis = j <= pos[r] && (a.window <= 0 || pos[r] - j < a.window);
            if (!vis) x = -INFINITY;
          }
          const float p = fast_exp2(x - lse2[r]);
          s[n][2 * r + e] = p * (dp[n][2 * r + e] - Dr[r]);   // s now holds dS
        }

    // ---- dq += dS K  (this warp's keys as the reduction dim: transposed loads)
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t a0 = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
      const uint32_t a1 = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
      const uint32_t a2 = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      const uint32_t a3 = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dpi = 0; dpi < 8; ++dpi) {
        const int row = kb0 + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int c = 2 * dpi + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(kb + swz(row, c), b0, b1, b2, b3);
        mma_bf16_16816(dq[2 * dpi], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816(dq[2 * dpi + 1], a0, a1, a2, a3, b2, b3);
      }
    }

    // ---- dr += (dS sheared to [row, distance]) . P_slice^T inside the band
    if (band) {
      // window column c holds distance cbw + c; row gq + 8r, key j0 + bcol sits
      // at column pos - j0 - bcol - cbw (always inside [0, 88) for this group)
      if (!use_rall) __syncthreads();    // both warps of the group read their R
      __nv_bfloat16 *dsw = reinterpret_cast<__nv_bfloat16 *>(win);
      for (int idx = 32 * kh + lane; idx < 16 * DSW / 8; idx += 64)
        reinterpret_cast<uint4 *>(dsw)[idx] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        __nv_bfloat16 *drow = dsw + (gq + 8 * r) * DSW + (pos[r] - j0 - cbw);
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            drow[-(kb0 + n * 8 + 2 * qq + e)] = __float2bfloat16_rn(s[n][2 * r + e]);
      }
      __syncthreads();
      // warp kh takes k16 steps [3 kh, 3 kh + 3) of the window's 6
#pragma unroll
      for (int ks = 0; ks < 3; ++ks) {
        const int kk = 3 * kh + ks;
        uint32_t wa[4];
        {
          const int row = (lane & 7) + (((lane >> 3) & 1) << 3);
          ldsm_x4_n(win_s + (row * DSW + kk * 16 + ((lane >> 4) << 3)) * 2, wa);
        }
        for (int np = 0; np < a.rd_pad / 16; ++np) {
          const int prow = np * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int pcol = coloff + kk * 16 + (((lane >> 3) & 1) << 3);
          uint32_t bq[4];
          ldsm_x4_n(pb + (prow * p_stride(PWQ) + pcol) * 2, bq);
          // (rd_pad / 16 is 1..4: the accumulator index spelled out per case)
          if (np == 0) { mma_bf16_16816(dr[0], wa[0], wa[1], wa[2], wa[3], bq[0], bq[1]);
                         mma_bf16_16816(dr[1], wa[0], wa[1], wa[2], wa[3], bq[2], bq[3]); }
          if (np == 1) { mma_bf16_16816(dr[2], wa[0], wa[1], wa[2], wa[3], bq[0], bq[1]);
                         mma_bf16_16816(dr[3], wa[0], wa[1], wa[2], wa[3], bq[2], bq[3]); }
          if (np == 2) { mma_bf16_16816(dr[4], wa[0], wa[1], wa[2], wa[3], bq[0], bq[1]);
                         mma_bf16_16816(dr[5], wa[0], wa[1], wa[2], wa[3], bq[2], bq[3]); }
          if (np == 3) { mma_bf16_16816(dr[6], wa[0], wa[1], wa[2], wa[3], bq[0], bq[1]);
                         mma_bf16_16816(dr[7], wa[0], wa[1], wa[2], wa[3], bq[2], bq[3]); }
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- the key-half 1 warps' partial dq / dr through shared memory (the K / V ring is free)
  float *part = reinterpret_cast<float *>(smem + L::kv);   // [4 groups][24 n8][4][32 lanes]
  if (kh == 1) {
#pragma unroll
    for (int n = 0; n < 16; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) part[((rw * 24) + n) * 128 + c * 32 + lane] = dq[n][c];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) part[((rw * 24) + 16 + n) * 128 + c * 32 + lane] = dr[n][c];
  }
  __syncthreads();
  if (kh == 1) return;
#pragma unroll
  for (int n = 0; n < 16; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) dq[n][c] += part[((rw * 24) + n) * 128 + c * 32 + lane];
#pragma unroll
  for (int n = 0; n < 8; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) dr[n][c] += part[((rw * 24) + 16 + n) * 128 + c * 32 + lane];

  // ---- epilogue: dq = s alpha acc, dr = s acc (bf16)
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int rl = rw * 16 + gq + 8 * r;
    if (rl >= nrows) continue;
    const size_t row = (size_t)(cq + row0 + rl) * a.Hq + h;
    const float fq = srow[r] * a.alpha;
    __nv_bfloat16 *dst = a.dq + row * kHeadDim + 2 * qq;
    const float *part = a.dq_split ? a.dq_part + row * kHeadDim + 2 * qq : nullptr;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      float x0 = dq[n][2 * r] * fq, x1 = dq[n][2 * r + 1] * fq;
      if (part) {
        const float2 pp = *reinterpret_cast<const float2 *>(part + n * 8);
        x0 += pp.x;
        x1 += pp.y;
      }
      *reinterpret_cast<uint32_t *>(dst + n * 8) = pack_bf16x2(x0, x1);
    }
    if (a.dr != nullptr) {
      __nv_bfloat16 *drd = a.dr + row * a.rd;
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = n * 8 + 2 * qq + e;
          if (c < a.rd) drd[c] = __float2bfloat16_rn(dr[n][2 * r + e] * srow[r]);
        }
    }
  }
}

// ------------------------------------------------------------------ dk / dv (key-major)

struct DkvLayout {
  static constexpr int k = 0;                               // K tile [64][128] swizzled
  static constexpr int v = k + BT * 256;                    // V tile
  static constexpr int rwin = v + BT * 256;                 // R window [64][RSK] fp32
  static constexpr int ring = rwin + BT * RSK * 4 + 128 - (BT * RSK * 4) % 128;
  // one stage: q, dout [64][128] swizzled; per-row lse2, D, s; r [64][rd_pad+8]; P slice
  static constexpr int s_q = 0, s_do = BT * 256, s_lse = 2 * BT * 256, s_d = s_lse + BT * 4,
                       s_sc = s_d + BT * 4, s_r = s_sc + BT * 4;
  __host__ __device__ static int r_stride(int rd_pad) { return (rd_pad + 8) * 2; }
  __host__ __device__ static int s_p(int rd_pad) { return s_r + BT * r_stride(rd_pad); }
  __host__ __device__ static int stage(int rd_pad) { return s_p(rd_pad) + rd_pad * p_stride(PWK) * 2; }
  __host__ __device__ static int total(int rd_pad) { return ring + BSTAGES * stage(rd_pad); }
};

__global__ void __launch_bounds__(NTB, 1) relattn_bwd_dkdv_kernel(const __grid_constant__ BwdArgs a) {
  using L = DkvLayout;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, qq = lane & 3;

  const int g = blockIdx.y, b = blockIdx.z;
  const int cq = a.cu_q[b], ck = a.cu_k[b];
  const int Lq = a.cu_q[b + 1] - cq, Lk = a.cu_k[b + 1] - ck;
  if (Lq < 0 || Lk < Lq || Lq > a.max_q || Lk > a.max_k) {
    if (tid == 0) atomicOr(a.err, kDevErrSeqlens);
    return;
  }
  const int j0 = blockIdx.x * BT;
  const int nkeys = min(BT, Lk - j0);
  if (nkeys <= 0) return;
  const int off = Lk - Lq;
  // query rows that see some key of the tile
  const int pos_hi = a.window > 0 ? min(Lk - 1, j0 + nkeys - 1 + a.window - 1) : Lk - 1;
  const int t_lo = max(0, j0 - off), t_hi = min(Lq - 1, pos_hi - off);
  const int qt_lo = t_lo / BT, n_qt = t_hi >= t_lo ? t_hi / BT - qt_lo + 1 : 0;
  const int npairs = a.group * n_qt;
  const bool has_bias = a.rd > 0 && a.E > 0;
  const int stage_bytes = L::stage(a.rd_pad);

  auto pair_h = [&](int it) { return g * a.group + it / n_qt; };
  auto pair_t0 = [&](int it) { return (qt_lo + it % n_qt) * BT; };
  auto is_band = [&](int t0) { return has_bias && (off + t0 - (j0 + BT - 1) < a.E); };

  auto issue_pair = [&](int it) {
    const int h = pair_h(it), t0 = pair_t0(it);
    const uint32_t sb = sbase + L::ring + (it % BSTAGES) * stage_bytes;
    uint8_t *sp = smem + L::ring + (it % BSTAGES) * stage_bytes;
    for (int idx = tid; idx < BT * 16; idx += NTB) {
      const int row = idx >> 4, c = idx & 15, t = t0 + row;
      const bool ok = t < Lq;
      const size_t gi = ((size_t)(cq + (ok ? t : 0)) * a.Hq + h) * kHeadDim + c * 8;
      cp_async16(sb + L::s_q + swz(row, c), a.q + gi, ok);
      cp_async16(sb + L::s_do + swz(row, c), a.dout + gi, ok);
    }
    if (tid < BT) {
      const int t = t0 + tid;
      const bool ok = t < Lq;
      const size_t li = (size_t)h * a.total_q + cq + (ok ? t : 0);
      reinterpret_cast<float *>(sp + L::s_lse)[tid] = ok ? a.lse[li] * kLog2e : INFINITY;
      reinterpret_cast<float *>(sp + L::s_d)[tid] = ok ? a.Dsum[li] : 0.f;
      reinterpret_cast<float *>(sp + L::s_sc)[tid] = log_scale(off + t, a.inv_ln_base);
    }
    if (is_band(t0)) {
      const int rcs = a.rd_pad / 8;
      for (int idx = tid; idx < BT * rcs; idx += NTB) {
        const int row = idx / rcs, c = idx - row * rcs, t = t0 + row;
        const bool ok = t < Lq && c * 8 < a.rd;
        const __nv_bfloat16 *src = a.r + ((size_t)(cq + (t < Lq ? t : 0)) * a.Hq + h) * a.rd;
        cp_async16(sb + L::s_r + row * L::r_stride(a.rd_pad) + c * 16, src + (ok ? c * 8 : 0), ok);
      }
      load_p_slice<PWK>(a, sb + L::s_p(a.rd_pad), floor8(off + t0 - j0 - (BT - 1)), tid);
    }
  };

  // K and V of the tile (keys past the end read as zero)
  for (int idx = tid; idx < BT * 16; idx += NTB) {
    const int row = idx >> 4, c = idx & 15, j = j0 + row;
    const bool ok = j < Lk;
    const size_t gi = ((size_t)(ck + (ok ? j : 0)) * a.Hkv + g) * kHeadDim + c * 8;
    cp_async16(sbase + L::k + swz(row, c), a.k + gi, ok);
    cp_async16(sbase + L::v + swz(row, c), a.v + gi, ok);
  }
#pragma unroll
  for (int s = 0; s < BSTAGES - 1; ++s) {
    if (s < npairs) issue_pair(s);
    cp_async_commit();
  }

  float dk[16][4], dv[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    dk[n][0] = dk[n][1] = dk[n][2] = dk[n][3] = 0.f;
    dv[n][0] = dv[n][1] = dv[n][2] = dv[n][3] = 0.f;
  }
  // warp (rw, kh): keys 16 rw .. 16 rw + 15 of the tile, query rows 32 kh .. 32 kh + 31
  // of each query tile; the two halves' dk / dv are summed at the end
  const int rw = warp & (NGRP - 1), kh = warp / NGRP;
  const int arow = rw * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);     // A-operand ldmatrix row
  int jk[2];                                                             // the thread's two keys
  jk[0] = j0 + rw * 16 + gq;
  jk[1] = jk[0] + 8;
  float *rwin = reinterpret_cast<float *>(smem + L::rwin);

  for (int it = 0; it < npairs; ++it) {
    cp_async_wait<BSTAGES - 2>();
    __syncthreads();
    if (it + BSTAGES - 1 < npairs) issue_pair(it + BSTAGES - 1);
    cp_async_commit();
    const int t0 = pair_t0(it);
    const int pos0 = off + t0;
    const uint32_t sb = sbase + L::ring + (it % BSTAGES) * stage_bytes;
    const float *lse2 = reinterpret_cast<const float *>(smem + L::ring + (it % BSTAGES) * stage_bytes + L::s_lse);
    const float *Dv = lse2 + BT;
    const float *scv = Dv + BT;
    const bool band = is_band(t0);
    const int cb = floor8(pos0 - j0 - (BT - 1));

    if (band) {
      // R window [64 query rows][136 distances from cb] = r . P_slice, fp32
      const uint32_t rb = sb + L::s_r;
      const uint32_t pb = sb + L::s_p(a.rd_pad);
      const int rstride = L::r_stride(a.rd_pad);
      // warp (rw, kh): rows 16 rw .. 16 rw + 15, n8 tiles [9 kh, 9 kh + 9) of the 17
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        constexpr int NH = 6;
        const int nt0 = 9 * kh + pass * NH, nt_end = min(9 * kh + 9, PWK / 8);
        float racc[NH][4];
#pragma unroll
        for (int n = 0; n < NH; ++n) racc[n][0] = racc[n][1] = racc[n][2] = racc[n][3] = 0.f;
        for (int kk = 0; kk < a.rd_pad / 16; ++kk) {
          uint32_t ra[4];
          ldsm_x4_n(rb + arow * rstride + (kk * 16 + ((lane >> 4) << 3)) * 2, ra);
          const int prow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
          for (int np = 0; np < NH / 2; ++np) {
            const int nt = nt0 + 2 * np;
            if (nt + 1 < nt_end) {
              uint32_t b0, b1, b2, b3;
              ldsm_x4_t(pb + (prow * p_stride(PWK) + nt * 8 + ((lane >> 4) << 3)) * 2, b0, b1, b2, b3);
              mma_bf16_16816(racc[2 * np], ra[0], ra[1], ra[2], ra[3], b0, b1);
              mma_bf16_16816(racc[2 * np + 1], ra[0], ra[1], ra[2], ra[3], b2, b3);
            } else if (nt < nt_end) {
              uint32_t b0, b1;
              ldsm_x2_t(pb + (prow * p_stride(PWK) + nt * 8) * 2, b0, b1);
              mma_bf16_16816(racc[2 * np], ra[0], ra[1], ra[2], ra[3], b0, b1);
            }
          }
        }
#pragma unroll
        for (int n = 0; n < NH; ++n) {
          const int nt = nt0 + n;
          if (nt < nt_end) {
            const int c = nt * 8 + 2 * qq;
            float *r0 = rwin + (rw * 16 + gq) * RSK + c;
            float *r1 = r0 + 8 * RSK;
            r0[0] = racc[n][0];
            r0[1] = racc[n][1];
            r1[0] = racc[n][2];
            r1[1] = racc[n][3];
          }
        }
      }
      __syncthreads();
    }

    const bool need_mask = (j0 + BT - 1 > pos0) ||
                           (a.window > 0 && j0 < pos0 + BT - 1 - a.window + 1) || (t0 + BT > Lq);
    {
      const int qc = 32 * kh;
      // ---- S^T = K_w Q^T and dP^T = V_w dout^T (16 keys x 32 queries)
      float st[4][4], dpt[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        st[n][0] = st[n][1] = st[n][2] = st[n][3] = 0.f;
        dpt[n][0] = dpt[n][1] = dpt[n][2] = dpt[n][3] = 0.f;
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t ka[4], va[4];
        ldsm_x4_n(sbase + L::k + swz(arow, 2 * kk + (lane >> 4)), ka);
        ldsm_x4_n(sbase + L::v + swz(arow, 2 * kk + (lane >> 4)), va);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const int row = qc + np * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int c = 2 * kk + ((lane >> 3) & 1);
          uint32_t qf[4], df[4];
          ldsm_x4_n(sb + L::s_q + swz(row, c), qf);
          ldsm_x4_n(sb + L::s_do + swz(row, c), df);
          mma_bf16_16816(st[2 * np], ka[0], ka[1], ka[2], ka[3], qf[0], qf[1]);
          mma_bf16_16816(st[2 * np + 1], ka[0], ka[1], ka[2], ka[3], qf[2], qf[3]);
          mma_bf16_16816(dpt[2 * np], va[0], va[1], va[2], va[3], df[0], df[1]);
          mma_bf16_16816(dpt[2 * np + 1], va[0], va[1], va[2], va[3], df[2], df[3]);
        }
      }
      // ---- P^T and dS^T (scaled by s_i alpha for dk)
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int il = qc + n * 8 + 2 * qq + e;            // query row in the tile
          const float sc = scv[il], l2 = lse2[il], Di = Dv[il];
          const int pos = pos0 + il;
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            float x = st[n][2 * rr + e] * a.alpha;
            if (band) {
              const int d = pos - jk[rr];
              x += rwin[il * RSK + d - cb];
            }
            x *= sc * kLog2e;
            if (need_mask) {
              const bool vis = jk[rr] <= pos && (a.window <= 0 || pos - jk[rr] < a.window);
              if (!vis) x = -INFINITY;
            }
            const float p = fast_exp2(x - l2);
            st[n][2 * rr + e] = p;
            dpt[n][2 * rr + e] = p * (dpt[n][2 * rr + e] - Di) * sc * a.alpha;
          }
        }
      // ---- dv += P^T dout, dk += dS^T q  (queries as the reduction dim)
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const uint32_t p0 = pack_bf16x2(st[2 * kk][0], st[2 * kk][1]);
        const uint32_t p1 = pack_bf16x2(st[2 * kk][2], st[2 * kk][3]);
        const uint32_t p2 = pack_bf16x2(st[2 * kk + 1][0], st[2 * kk + 1][1]);
        const uint32_t p3 = pack_bf16x2(st[2 * kk + 1][2], st[2 * kk + 1][3]);
        const uint32_t s0 = pack_bf16x2(dpt[2 * kk][0], dpt[2 * kk][1]);
        const uint32_t s1 = pack_bf16x2(dpt[2 * kk][2], dpt[2 * kk][3]);
        const uint32_t s2 = pack_bf16x2(dpt[2 * kk + 1][0], dpt[2 * kk + 1][1]);
        const uint32_t s3 = pack_bf16x2(dpt[2 * kk + 1][2], dpt[2 * kk + 1][3]);
#pragma unroll
        for (int dpi = 0; dpi < 8; ++dpi) {
          const int row = qc + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int c = 2 * dpi + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sb + L::s_do + swz(row, c), b0, b1, b2, b3);
          mma_bf16_16816(dv[2 * dpi], p0, p1, p2, p3, b0, b1);
          mma_bf16_16816(dv[2 * dpi + 1], p0, p1, p2, p3, b2, b3);
          ldsm_x4_t(sb + L::s_q + swz(row, c), b0, b1, b2, b3);
          mma_bf16_16816(dk[2 * dpi], s0, s1, s2, s3, b0, b1);
          mma_bf16_16816(dk[2 * dpi + 1], s0, s1, s2, s3, b2, b3);
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- the second half's partial dk / dv through shared memory (the ring is free)
  float *part = reinterpret_cast<float *>(smem + L::ring);   // [4 groups][2][16 n8][4][32 lanes]
  if (kh == 1) {
#pragma unroll
    for (int n = 0; n < 16; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        part[((rw * 2 + 0) * 64 + n * 4 + c) * 32 + lane] = dk[n][c];
        part[((rw * 2 + 1) * 64 + n * 4 + c) * 32 + lane] = dv[n][c];
      }
  }
  __syncthreads();
  if (kh == 1) return;
#pragma unroll
  for (int n = 0; n < 16; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      dk[n][c] += part[((rw * 2 + 0) * 64 + n * 4 + c) * 32 + lane];
      dv[n][c] += part[((rw * 2 + 1) * 64 + n * 4 + c) * 32 + lane];
    }

  // ---- epilogue (keys of the tile that no query sees get zeros)
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int kl = rw * 16 + gq + 8 * rr;
    if (kl >= nkeys) continue;
    const size_t row = (size_t)(ck + j0 + kl) * a.Hkv + g;
    __nv_bfloat16 *dkd = a.dk + row * kHeadDim + 2 * qq;
    __nv_bfloat16 *dvd = a.dv + row * kHeadDim + 2 * qq;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      *reinterpret_cast<uint32_t *>(dkd + n * 8) = pack_bf16x2(dk[n][2 * rr], dk[n][2 * rr + 1]);
      *reinterpret_cast<uint32_t *>(dvd + n * 8) = pack_bf16x2(dv[n][2 * rr], dv[n][2 * rr + 1]);
    }
  }
}

}  // namespace

size_t bwd_dq_smem_bytes(int rd_pad) { return DqLayout::total(rd_pad); }
size_t bwd_dkdv_smem_bytes(int rd_pad) { return DkvLayout::total(rd_pad); }

cudaError_t launch_backward(const BwdArgs &a, int sms, cudaStream_t stream) {
  const bool tc = bwd_tc_supported(a);
  if (tc && a.rd > 0 && a.E > 0) {   // R = r . P for every row, read by the tcgen05 dk / dv
    const int smem = RPT * (a.rd_pad + 8) * 2 + a.rd_pad * p_stride(RPT) * 2;
    const long rows = (long)a.total_q * a.Hq;
    relattn_bwd_rel_kernel<<<(unsigned)((rows + RPT - 1) / RPT), 256, smem, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    const long rows = (long)a.total_q * a.Hq;
    long blocks = (rows * 16 + 255) / 256;
    const long cap = (long)(sms > 0 ? sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks > 0) relattn_bwd_dot_kernel<<<(unsigned)blocks, 256, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // dq: on tcgen05 over the keys outside the bias band (all keys without a
  // bias); the band's keys, and every key when tcgen05 is unavailable, on
  // the warp-MMA kernel, which adds the tcgen05 part
  const bool bias = a.rd > 0 && a.E > 0;
  const bool tcq = tc && bwd_dq_tc_supported(a);
  BwdArgs aq = a;
  aq.dq_split = tcq && bias ? 1 : 0;
  aq.rall_ok = tc && bias ? 1 : 0;       // the pre-pass above ran
  if (tcq) {
    cudaError_t e = launch_bwd_dq_tc(aq, stream);
    if (e != cudaSuccess) return e;
    if (!bias && a.dr != nullptr &&   // r without an extent: dr is zero, and no kernel below writes it
        (e = cudaMemsetAsync(a.dr, 0, (size_t)a.total_q * a.Hq * a.rd * sizeof(__nv_bfloat16), stream)) !=
            cudaSuccess)
      return e;
  }
  if (!tcq || bias) {
    const int smem = (int)DqLayout::total(a.rd_pad);
    cudaError_t e = cudaFuncSetAttribute(relattn_bwd_dq_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    relattn_bwd_dq_kernel<<<dim3(a.q_tiles, a.Hq, a.batch), NTB, smem, stream>>>(aq);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (tc) return launch_bwd_dkdv_tc(a, stream);
  {
    const int smem = (int)DkvLayout::total(a.rd_pad);
    cudaError_t e = cudaFuncSetAttribute(relattn_bwd_dkdv_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    relattn_bwd_dkdv_kernel<<<dim3(a.k_tiles, a.Hkv, a.batch), NTB, smem, stream>>>(a);
    return cudaGetLastError();
  }
}

}  // namespace relattn
