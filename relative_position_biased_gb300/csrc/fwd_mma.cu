// fwd_mma.cu -- relative-attention forward on warp-level bf16 MMAs
// (mma.sync m16n8k16), shared by prefill and split-KV decode.
//
// What one CTA computes (page "SGLang and Miles Add Day-0 Support for
// Inkling", section "Attention with Relative Positional Embedding"):
// for a block of query rows (t, h) and a range of keys j,
//     x(t,h,j) = s(i) * (alpha * q.k + [0 <= i-j < E] * r_{t,h} . P[:, i-j])
// followed by an online (running max / running sum) softmax and the PV
// product.  The relative bias is added inside the online softmax, as the FA4
// fork on that page does ("Relative Logits Optimization", Figure 3), but the
// sheared bias is never materialised in global memory: for every key tile
// inside the bias band each warp multiplies its 16 rows of r by the slice of P
// covering the distances it can see (a 16 x 88 x r_dim MMA), parks that small
// R window in shared memory, and each score gathers R[row][i - j - base].
// Tiles wholly past the band, or wholly inside the causal/window range, skip
// the gather or the mask respectively; tiles outside the range are never
// visited.
//
// Data movement: K/V tiles of 64 keys x 128 dims (bf16, 256 B rows, 16-byte
// chunks XOR-swizzled by row) and the P slice of each band tile are streamed
// into a multi-stage cp.async ring; Q and r are loaded once per CTA.
#include "launch.h"

namespace relattn {
namespace {

constexpr int BN = 64;    // keys per tile
constexpr int RW = 88;    // R window columns per warp (11 n8 tiles)
constexpr int RWS = 88;   // fp32 row stride of a warp's R window

template <int NW, int STAGES, int PW>
struct Layout {
  static constexpr int M = NW * 16;          // query rows per CTA
  static constexpr int PS = PW + 8;          // bf16 row stride of a P slice
  static constexpr int q_bytes = M * 256;    // Q tile; later reused for R windows
  static constexpr int rwin_bytes = NW * 16 * RWS * 4;
  static constexpr int region0 = q_bytes > rwin_bytes ? q_bytes : rwin_bytes;
  static constexpr int kv_stage = BN * 256;
  static constexpr int off_k = region0;
  static constexpr int off_v = off_k + STAGES * kv_stage;
  static constexpr int off_p = off_v + STAGES * kv_stage;
  __host__ __device__ static int p_stage(int rd_pad) { return rd_pad * PS * 2; }
  __host__ __device__ static int off_r(int rd_pad) { return off_p + STAGES * p_stage(rd_pad); }
  __host__ __device__ static int r_stride(int rd_pad) { return (rd_pad + 8) * 2; }
  __host__ __device__ static int total(int rd_pad) { return off_r(rd_pad) + M * r_stride(rd_pad); }
};

__device__ __forceinline__ int floor8(int x) { return x & ~7; }

template <bool DECODE, int NW, int STAGES, int PW>
__global__ void __launch_bounds__(NW * 32, 1) relattn_fwd_mma_kernel(const __grid_constant__ KernelArgs a) {
  using L = Layout<NW, STAGES, PW>;
  constexpr int M = L::M;
  constexpr int NT = NW * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, qq = lane & 3;

  // ------------------------------------------------------------ work item
  int b, head, split = 0, row_block = 0, q_tile = 0;
  if (DECODE) {
    split = blockIdx.x;
    head = blockIdx.y / a.row_blocks;      // kv head
    row_block = blockIdx.y % a.row_blocks;
    b = blockIdx.z;
  } else {
    q_tile = a.q_tiles - 1 - blockIdx.x;   // longest-running tiles first
    head = blockIdx.y;                     // query head
    b = blockIdx.z;
  }
  const int cq = a.cu_q[b], ck = a.cu_k[b];
  const int Lq = a.cu_q[b + 1] - cq, Lk = a.cu_k[b + 1] - ck;
  if (Lq < 0 || Lk < Lq || Lq > a.max_q || Lk > a.max_k) {
    if (tid == 0) atomicOr(a.err, kDevErrSeqlens);
    return;
  }
  const int off = Lk - Lq;  // bottom-right alignment
  const int row0 = DECODE ? row_block * M : q_tile * M;
  const int nrows = min(M, (DECODE ? Lq * a.group : Lq) - row0);
  if (nrows <= 0) return;
  const int kv_head = DECODE ? head : head / a.group;

  // row (local, clamped to the last valid row) -> (t, h)
  auto row_t = [&](int rl) {
    const int x = row0 + min(rl, nrows - 1);
    return DECODE ? x / a.group : x;
  };
  auto row_h = [&](int rl) {
    const int x = row0 + min(rl, nrows - 1);
    return DECODE ? head * a.group + x % a.group : head;
  };

  const int p_min = off + row_t(0), p_max = off + row_t(nrows - 1);
  const int j_lo = a.window > 0 ? max(0, p_min - a.window + 1) : 0;
  int kbeg = j_lo & ~(BN - 1), kend = p_max + 1;
  if (DECODE) {
    kbeg += split * a.split_chunk;
    kend = min(kend, kbeg + a.split_chunk);
  }
  const int ntiles = kend > kbeg ? (kend - kbeg + BN - 1) / BN : 0;
  auto tile_j0 = [&](int it) { return kbeg + (ntiles - 1 - it) * BN; };  // diagonal first

  const bool has_bias = a.rd > 0 && a.E > 0;
  auto is_band = [&](int j0) { return has_bias && (p_min - (j0 + BN - 1) < a.E); };

  // ------------------------------------------------------------ loaders
  auto load_kv = [&](int j0, int stage) {
    for (int idx = tid; idx < BN * 16; idx += NT) {
      const int row = idx >> 4, c = idx & 15, j = j0 + row;
      const bool ok = j < Lk;
      const size_t g = ((size_t)(ck + (ok ? j : 0)) * a.Hkv + kv_head) * kHeadDim + c * 8;
      const uint32_t sw = row * 256 + ((c ^ (row & 7)) << 4);
      cp_async16(sbase + L::off_k + stage * L::kv_stage + sw, a.k + g, ok);
      cp_async16(sbase + L::off_v + stage * L::kv_stage + sw, a.v + g, ok);
    }
  };
  // P columns [cb, cb + PW) for all rd_pad channels; out-of-range -> 0.
  auto load_p = [&](int j0, int stage) {
    const int cb = floor8(p_min - j0 - BN);
    constexpr int cpr = PW / 8;
    const uint32_t base = sbase + L::off_p + stage * L::p_stage(a.rd_pad);
    for (int idx = tid; idx < a.rd_pad * cpr; idx += NT) {
      const int c = idx / cpr, x = idx - c * cpr, col = cb + x * 8;
      const uint32_t dst = base + (c * L::PS + x * 8) * 2;
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
          const __nv_bfloat16 z = __float2bfloat16(0.f);
          __nv_bfloat16 lo = (in_row && c0 >= 0 && c0 < a.E) ? a.P[(size_t)c * a.E + c0] : z;
          __nv_bfloat16 hi = (in_row && c1 >= 0 && c1 < a.E) ? a.P[(size_t)c * a.E + c1] : z;
          w[e] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
        }
        st_shared_v4(dst, w[0], w[1], w[2], w[3]);
      }
    }
  };
  auto issue_tile = [&](int it) {
    const int j0 = tile_j0(it), stage = it % STAGES;
    load_kv(j0, stage);
    if (is_band(j0)) load_p(j0, stage);
  };

  // Q rows (swizzled like K) and r rows (padded stride) -- first async group.
  for (int idx = tid; idx < M * 16; idx += NT) {
    const int row = idx >> 4, c = idx & 15;
    const size_t g = ((size_t)(cq + row_t(row)) * a.Hq + row_h(row)) * kHeadDim + c * 8;
    cp_async16(sbase + row * 256 + ((c ^ (row & 7)) << 4), a.q + g, true);
  }
  if (has_bias) {
    const int rcs = a.rd_pad / 8;
    const uint32_t rb = sbase + L::off_r(a.rd_pad);
    for (int idx = tid; idx < M * rcs; idx += NT) {
      const int row = idx / rcs, c = idx - row * rcs;
      const __nv_bfloat16 *src = a.r + ((size_t)(cq + row_t(row)) * a.Hq + row_h(row)) * a.rd;
      const uint32_t dst = rb + row * L::r_stride(a.rd_pad) + c * 16;
      if (a.r_vec_ok) {
        cp_async16(dst, src + (c * 8 < a.rd ? c * 8 : 0), c * 8 < a.rd);
      } else {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c0 = c * 8 + 2 * e;
          const unsigned short lo = c0 < a.rd ? __bfloat16_as_ushort(src[c0]) : 0;
          const unsigned short hi = c0 + 1 < a.rd ? __bfloat16_as_ushort(src[c0 + 1]) : 0;
          w[e] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        st_shared_v4(dst, w[0], w[1], w[2], w[3]);
      }
    }
  }
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < ntiles) issue_tile(s);
    cp_async_commit();
  }

  // ------------------------------------------------------------ per-row state
  float cqk[2], cbias[2];
  int pos[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int rl = warp * 16 + gq + 8 * r;
    pos[r] = off + row_t(rl);
    const float sc = log_scale(pos[r], a.inv_ln_base);
    cqk[r] = a.alpha_log2e * sc;
    cbias[r] = kLog2e * sc;
  }
  const int p_w0 = off + row_t(warp * 16);

  uint32_t qa[8][4];
  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  float *rwin = reinterpret_cast<float *>(smem) + warp * 16 * RWS;

  for (int it = 0; it < ntiles; ++it) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    if (it == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int row = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int c = 2 * kk + (lane >> 4);
        ldsm_x4(sbase + row * 256 + ((c ^ (row & 7)) << 4), qa[kk][0], qa[kk][1], qa[kk][2],
                qa[kk][3]);
      }
      __syncthreads();  // region 0 now holds the R windows
    }
    if (it + STAGES - 1 < ntiles) issue_tile(it + STAGES - 1);
    cp_async_commit();

    const int stage = it % STAGES, j0 = tile_j0(it);
    // ---- S = Q K^T
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
    const uint32_t kb = sbase + L::off_k + stage * L::kv_stage;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int row = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = 2 * kk + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + row * 256 + ((c ^ (row & 7)) << 4), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
        mma_bf16_16816(s[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
      }
    }

    // ---- relative bias: R window = r_rows . P[:, cbw .. cbw+88), gathered per score
    const bool band = is_band(j0);
    if (band) {
      const int cb = floor8(p_min - j0 - BN);
      const int cbw = floor8(p_w0 - j0 - BN);
      const int coloff = cbw - cb;
      const uint32_t pb = sbase + L::off_p + stage * L::p_stage(a.rd_pad);
      const uint32_t rb = sbase + L::off_r(a.rd_pad);
      const int rstride = L::r_stride(a.rd_pad);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        constexpr int NH0 = 6;                 // n8 tiles in the first pass
        const int nt0 = half ? NH0 : 0;
        float racc[NH0][4];
#pragma unroll
        for (int n = 0; n < NH0; ++n) racc[n][0] = racc[n][1] = racc[n][2] = racc[n][3] = 0.f;
        for (int kk = 0; kk < a.rd_pad / 16; ++kk) {
          uint32_t a0, a1, a2, a3;
          {
            const int row = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int col = kk * 16 + ((lane >> 4) << 3);
            ldsm_x4(rb + row * rstride + col * 2, a0, a1, a2, a3);
          }
          const int prow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
          for (int np = 0; np < NH0 / 2; ++np) {
            const int nt = nt0 + 2 * np;
            if (nt + 1 < RW / 8) {
              const int pcol = coloff + nt * 8 + ((lane >> 4) << 3);
              uint32_t b0, b1, b2, b3;
              ldsm_x4_t(pb + (prow * L::PS + pcol) * 2, b0, b1, b2, b3);
              mma_bf16_16816(racc[2 * np], a0, a1, a2, a3, b0, b1);
              mma_bf16_16816(racc[2 * np + 1], a0, a1, a2, a3, b2, b3);
            } else if (nt < RW / 8) {
              const int pcol = coloff + nt * 8;
              uint32_t b0, b1;
              ldsm_x2_t(pb + (prow * L::PS + pcol) * 2, b0, b1);
              mma_bf16_16816(racc[2 * np], a0, a1, a2, a3, b0, b1);
            }
          }
        }
#pragma unroll
        for (int n = 0; n < NH0; ++n) {
          const int nt = nt0 + n;
          if (nt < RW / 8) {
            *reinterpret_cast<float2 *>(&rwin[gq * RWS + nt * 8 + 2 * qq]) =
                make_float2(racc[n][0], racc[n][1]);
            *reinterpret_cast<float2 *>(&rwin[(gq + 8) * RWS + nt * 8 + 2 * qq]) =
                make_float2(racc[n][2], racc[n][3]);
          }
        }
      }
      __syncwarp();
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float *rrow = rwin + (gq + 8 * r) * RWS + (pos[r] - j0 - cbw);
#pragma unroll
        for (int n = 0; n < 8; ++n) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int bcol = n * 8 + 2 * qq + e;
            s[n][2 * r + e] = fmaf(s[n][2 * r + e], cqk[r], rrow[-bcol] * cbias[r]);
          }
        }
      }
      __syncwarp();
    } else {
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        s[n][0] *= cqk[0];
        s[n][1] *= cqk[0];
        s[n][2] *= cqk[1];
        s[n][3] *= cqk[1];
      }
    }

    // ---- mask (diagonal / window edge / sequence end tiles only)
    const bool need_mask = (j0 + BN - 1 > p_min) ||
                           (a.window > 0 && j0 < p_max - a.window + 1) || (j0 + BN > Lk);
    if (need_mask) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
#pragma unroll
        for (int n = 0; n < 8; ++n) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = j0 + n * 8 + 2 * qq + e;
            const bool vis = j <= pos[r] && (a.window <= 0 || pos[r] - j < a.window);
            if (!vis) s[n][2 * r + e] = -INFINITY;
          }
        }
      }
    }

    // ---- online softmax (base 2)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mx = -INFINITY;
#pragma unroll
      for (int n = 0; n < 8; ++n) mx = fmaxf(mx, fmaxf(s[n][2 * r], s[n][2 * r + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_r[r], mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float corr = fast_exp2(m_r[r] - m_use);
      m_r[r] = m_new;
      float rs = 0.f;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        s[n][2 * r] = fast_exp2(s[n][2 * r] - m_use);
        s[n][2 * r + 1] = fast_exp2(s[n][2 * r + 1] - m_use);
        rs += s[n][2 * r] + s[n][2 * r + 1];
      }
      l_r[r] = l_r[r] * corr + rs;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        o[n][2 * r] *= corr;
        o[n][2 * r + 1] *= corr;
      }
    }

    // ---- O += P V
    const uint32_t vb = sbase + L::off_v + stage * L::kv_stage;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t pa0 = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
      const uint32_t pa1 = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
      const uint32_t pa2 = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      const uint32_t pa3 = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        const int row = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int c = 2 * dp + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + row * 256 + ((c ^ (row & 7)) << 4), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], pa0, pa1, pa2, pa3, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa0, pa1, pa2, pa3, b2, b3);
      }
    }
  }
  cp_async_wait<0>();

  // ------------------------------------------------------------ epilogue
  const bool final_out = !DECODE || a.num_splits == 1;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float l = l_r[r];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const int rl = warp * 16 + gq + 8 * r;
    if (rl >= nrows) continue;
    const int t = row_t(rl), h = row_h(rl);
    const size_t row = (size_t)(cq + t) * a.Hq + h;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse = l > 0.f ? (m_r[r] + __log2f(l)) * kLn2 : -INFINITY;
    if (final_out) {
      __nv_bfloat16 *dst = a.out + row * kHeadDim + 2 * qq;
#pragma unroll
      for (int n = 0; n < 16; ++n)
        *reinterpret_cast<uint32_t *>(dst + n * 8) = pack_bf16x2(o[n][2 * r] * inv, o[n][2 * r + 1] * inv);
      if (qq == 0) a.lse[(size_t)h * a.total_q + cq + t] = lse;
    } else {
      const size_t prow = (size_t)split * a.total_q * a.Hq + row;
      float *dst = a.o_part + prow * kHeadDim + 2 * qq;
#pragma unroll
      for (int n = 0; n < 16; ++n)
        *reinterpret_cast<float2 *>(dst + n * 8) = make_float2(o[n][2 * r] * inv, o[n][2 * r + 1] * inv);
      if (qq == 0) a.lse_part[prow] = lse;
    }
  }
}

constexpr int kPrefillWarps = 8, kPrefillStages = 2, kPrefillPW = 208;
constexpr int kDecodeStages = 3, kDecodePW = 112;

template <bool DECODE, int NW, int STAGES, int PW>
cudaError_t launch_impl(const KernelArgs &a, dim3 grid, cudaStream_t stream) {
  using L = Layout<NW, STAGES, PW>;
  const int smem = L::total(a.rd_pad);
  auto kern = relattn_fwd_mma_kernel<DECODE, NW, STAGES, PW>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, NW * 32, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

int decode_warps_for_rows(int rows) {
  const int w = (rows + 15) / 16;
  if (w <= 1) return 1;
  if (w <= 2) return 2;
  if (w <= 4) return 4;
  if (w <= 5) return 5;
  return 8;
}

size_t prefill_mma_smem_bytes(int rd_pad) {
  return Layout<kPrefillWarps, kPrefillStages, kPrefillPW>::total(rd_pad);
}

size_t decode_mma_smem_bytes(int warps, int rd_pad) {
  switch (warps) {
    case 1: return Layout<1, kDecodeStages, kDecodePW>::total(rd_pad);
    case 2: return Layout<2, kDecodeStages, kDecodePW>::total(rd_pad);
    case 4: return Layout<4, kDecodeStages, kDecodePW>::total(rd_pad);
    case 5: return Layout<5, kDecodeStages, kDecodePW>::total(rd_pad);
    default: return Layout<8, kDecodeStages, kDecodePW>::total(rd_pad);
  }
}

cudaError_t launch_prefill_mma(const KernelArgs &a, cudaStream_t stream) {
  dim3 grid(a.q_tiles, a.Hq, a.batch);
  return launch_impl<false, kPrefillWarps, kPrefillStages, kPrefillPW>(a, grid, stream);
}

cudaError_t launch_decode_mma(const KernelArgs &a, int warps, cudaStream_t stream) {
  dim3 grid(a.num_splits, a.Hkv * a.row_blocks, a.batch);
  switch (warps) {
    case 1: return launch_impl<true, 1, kDecodeStages, kDecodePW>(a, grid, stream);
    case 2: return launch_impl<true, 2, kDecodeStages, kDecodePW>(a, grid, stream);
    case 4: return launch_impl<true, 4, kDecodeStages, kDecodePW>(a, grid, stream);
    case 5: return launch_impl<true, 5, kDecodeStages, kDecodePW>(a, grid, stream);
    case 8: return launch_impl<true, 8, kDecodeStages, kDecodePW>(a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace relattn
