// prologue.cu -- the attention prologue: K / V ShortConv, Q / K RMSNorm and
// the KV-cache write, in one pass over the chunk's rows.
//
// Page "SGLang and Miles Add Day-0 Support for Inkling": section "Short
// Convolution (ShortConv)" gives the filter, y[t,c] = x[t,c] + sum_{d=0}^{3}
// w[c,d] x[t-d,c] per channel over the token dimension; section "ShortConv
// Optimization", paragraph "KV ShortConv + QK-norm + KV store", fuses the
// K / V convolution, the Q / K RMSNorm and the cache write into one kernel.
//
// HBM bound: each (token, head) row of q, k and v is read once and written
// once (the three earlier rows a conv tap reads were just read by nearby
// warps, so they come from L2).  A warp takes 4 consecutive rows of the
// (token, slot) order -- slots are the q heads, then the k heads, then the v
// heads of a token -- and each lane 4 dims (8-byte accesses, 256 contiguous
// bytes per row); all loads of the 4 rows are issued before any arithmetic.
#include "launch.h"

namespace relattn {
namespace {

constexpr int kTaps = 4;            // W in the ShortConv equation
constexpr int kRowsPerWarp = 4;
constexpr int kPrologueThreads = 256;

struct PrologueArgs {
  const __nv_bfloat16 *q, *k, *v;
  const float *conv_k, *conv_v, *norm_q, *norm_k;
  float eps;
  const int32_t *cu_q, *cu_k;
  int batch, total_q, total_k, Hq, Hkv;
  __nv_bfloat16 *q_out, *k_cache, *v_cache;
  const __nv_bfloat16 *state_in_k, *state_in_v;
  __nv_bfloat16 *state_out_k, *state_out_v;
  int *err;
};

__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float (&x)[4]) {
  const uint2 u = *reinterpret_cast<const uint2 *>(p);
  x[0] = __uint_as_float(u.x << 16);
  x[1] = __uint_as_float(u.x & 0xffff0000u);
  x[2] = __uint_as_float(u.y << 16);
  x[3] = __uint_as_float(u.y & 0xffff0000u);
}

__device__ __forceinline__ void store4(__nv_bfloat16 *p, const float (&y)[4]) {
  uint2 u;
  u.x = pack_bf16x2(y[0], y[1]);
  u.y = pack_bf16x2(y[2], y[3]);
  *reinterpret_cast<uint2 *>(p) = u;
}

// sequence of a chunk row (cu_q ascending): last b with cu_q[b] <= row
__device__ __forceinline__ int seq_of(const int32_t *cu_q, int batch, int row) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_q[mid] <= row) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kPrologueThreads)
relattn_prologue_kernel(const PrologueArgs a) {
  const int lane = threadIdx.x & 31;
  const int slots = a.Hq + 2 * a.Hkv;
  const long rows = (long)a.total_q * slots;
  const long warps = (long)gridDim.x * (kPrologueThreads / 32);
  const int dim = 4 * lane;
  for (long r0 = ((long)blockIdx.x * (kPrologueThreads / 32) + (threadIdx.x >> 5)) * kRowsPerWarp;
       r0 < rows; r0 += warps * kRowsPerWarp) {
    // ---- loads of up to 4 rows: x[j][0] is the row itself, x[j][d] the
    // input d rows earlier in its sequence (conv rows only)
    float x[kRowsPerWarp][kTaps][4];
    int kind[kRowsPerWarp], head[kRowsPerWarp];
    long out_row[kRowsPerWarp];   // q row or cache row; -1: nothing to do
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) {
      const long r = r0 + j;
      out_row[j] = -1;
      kind[j] = 0;
      head[j] = 0;
      if (r >= rows) continue;
      const int t = (int)(r / slots), s = (int)(r - (long)t * slots);
      if (s < a.Hq) {                                       // q head s
        kind[j] = 0;
        head[j] = s;
        load4(a.q + ((size_t)t * a.Hq + s) * kHeadDim + dim, x[j][0]);
        out_row[j] = t;
        continue;
      }
      const bool is_k = s < a.Hq + a.Hkv;
      const int h = is_k ? s - a.Hq : s - a.Hq - a.Hkv;
      kind[j] = is_k ? 1 : 2;
      head[j] = h;
      const int b = seq_of(a.cu_q, a.batch, t);
      const int cq = a.cu_q[b], ck = a.cu_k[b];
      const int Lq = a.cu_q[b + 1] - cq, Lk = a.cu_k[b + 1] - ck;
      const int tc = t - cq;                                // row within the chunk
      // the row must lie in its sequence and the sequence's cache rows in the cache
      if (tc < 0 || tc >= Lq || Lk < Lq || ck < 0 || a.cu_k[b + 1] > a.total_k) {
        if (lane == 0) atomicOr(a.err, kDevErrSeqlens);
        continue;
      }
      const __nv_bfloat16 *src = is_k ? a.k : a.v;
      const __nv_bfloat16 *st = is_k ? a.state_in_k : a.state_in_v;
#pragma unroll
      for (int d = 0; d < kTaps; ++d) {
        const int p = tc - d;
        if (p >= 0) {
          load4(src + ((size_t)(cq + p) * a.Hkv + h) * kHeadDim + dim, x[j][d]);
        } else if (st != nullptr) {
          load4(st + ((size_t)b * (kTaps - 1) + (kTaps - 1 + p)) * a.Hkv * kHeadDim + h * kHeadDim + dim,
                x[j][d]);
        } else {
          x[j][d][0] = x[j][d][1] = x[j][d][2] = x[j][d][3] = 0.f;
        }
      }
      out_row[j] = (long)ck + (Lk - Lq) + tc;
    }
    // ---- arithmetic and stores
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) {
      if (out_row[j] < 0) continue;                        // (warp-uniform)
      float y[4];
      if (kind[j] == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) y[i] = x[j][0][i];
      } else {
        const float *w = (kind[j] == 1 ? a.conv_k : a.conv_v) + (size_t)(head[j] * kHeadDim + dim) * kTaps;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 wi = *reinterpret_cast<const float4 *>(w + i * kTaps);
          float acc = x[j][0][i];                           // the input added back
          acc = fmaf(wi.x, x[j][0][i], acc);
          acc = fmaf(wi.y, x[j][1][i], acc);
          acc = fmaf(wi.z, x[j][2][i], acc);
          acc = fmaf(wi.w, x[j][3][i], acc);
          y[i] = acc;
        }
      }
      if (kind[j] != 2) {                                   // RMSNorm (q, and k after its conv)
        float ss = y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = rsqrtf(ss * (1.f / kHeadDim) + a.eps);
        const float4 g = *reinterpret_cast<const float4 *>((kind[j] == 0 ? a.norm_q : a.norm_k) + dim);
        y[0] *= inv * g.x;
        y[1] *= inv * g.y;
        y[2] *= inv * g.z;
        y[3] *= inv * g.w;
      }
      __nv_bfloat16 *dst = kind[j] == 0 ? a.q_out + ((size_t)out_row[j] * a.Hq + head[j]) * kHeadDim
                           : (kind[j] == 1 ? a.k_cache : a.v_cache) +
                                 ((size_t)out_row[j] * a.Hkv + head[j]) * kHeadDim;
      store4(dst + dim, y);
    }
  }
}

// conv state after the chunk: the last 3 pre-convolution inputs of each
// sequence (from the chunk, else from the state before it, else zero)
__global__ void __launch_bounds__(kPrologueThreads)
relattn_prologue_state_kernel(const PrologueArgs a) {
  const int C = a.Hkv * kHeadDim;
  const long n = (long)a.batch * (kTaps - 1) * (C / 4);
  for (long e = (long)blockIdx.x * blockDim.x + threadIdx.x; e < 2 * n; e += (long)gridDim.x * blockDim.x) {
    const bool is_k = e < n;
    const long f = is_k ? e : e - n;
    const int c4 = (int)(f % (C / 4)), jb = (int)(f / (C / 4));
    const int j = jb % (kTaps - 1), b = jb / (kTaps - 1);
    const int cq = a.cu_q[b], Lq = a.cu_q[b + 1] - cq;
    if (cq < 0 || Lq < 0 || a.cu_q[b + 1] > a.total_q) {
      atomicOr(a.err, kDevErrSeqlens);
      continue;
    }
    const int p = Lq - (kTaps - 1) + j;                   // chunk row of state slot j
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    const __nv_bfloat16 *src = is_k ? a.k : a.v;
    const __nv_bfloat16 *st = is_k ? a.state_in_k : a.state_in_v;
    if (p >= 0) load4(src + (size_t)(cq + p) * C + 4 * c4, x);
    else if (st != nullptr) load4(st + ((size_t)b * (kTaps - 1) + (kTaps - 1 + p)) * C + 4 * c4, x);
    __nv_bfloat16 *dst = is_k ? a.state_out_k : a.state_out_v;
    if (dst != nullptr) store4(dst + ((size_t)b * (kTaps - 1) + j) * C + 4 * c4, x);
  }
}

}  // namespace

cudaError_t launch_prologue(const relattn_prologue_params *p, int *err, int sms, cudaStream_t stream) {
  PrologueArgs a;
  a.q = static_cast<const __nv_bfloat16 *>(p->q);
  a.k = static_cast<const __nv_bfloat16 *>(p->k);
  a.v = static_cast<const __nv_bfloat16 *>(p->v);
  a.conv_k = p->conv_k;
  a.conv_v = p->conv_v;
  a.norm_q = p->norm_q;
  a.norm_k = p->norm_k;
  a.eps = p->eps;
  a.cu_q = p->cu_seqlens_q;
  a.cu_k = p->cu_seqlens_k;
  a.batch = p->batch;
  a.total_q = p->total_q;
  a.total_k = p->total_k;
  a.Hq = p->num_heads_q;
  a.Hkv = p->num_heads_kv;
  a.q_out = static_cast<__nv_bfloat16 *>(p->q_out);
  a.k_cache = static_cast<__nv_bfloat16 *>(p->k_cache);
  a.v_cache = static_cast<__nv_bfloat16 *>(p->v_cache);
  a.state_in_k = static_cast<const __nv_bfloat16 *>(p->conv_state_in_k);
  a.state_in_v = static_cast<const __nv_bfloat16 *>(p->conv_state_in_v);
  a.state_out_k = static_cast<__nv_bfloat16 *>(p->conv_state_out_k);
  a.state_out_v = static_cast<__nv_bfloat16 *>(p->conv_state_out_v);
  a.err = err;
  const long rows = (long)a.total_q * (a.Hq + 2 * a.Hkv);
  if (rows > 0) {
    const long per_block = (long)(kPrologueThreads / 32) * kRowsPerWarp;
    long blocks = (rows + per_block - 1) / per_block;
    const long cap = (long)(sms > 0 ? sms : 148) * 8;   // 8 resident blocks per SM, grid-stride beyond
    if (blocks > cap) blocks = cap;
    relattn_prologue_kernel<<<(unsigned)blocks, kPrologueThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.state_out_k != nullptr || a.state_out_v != nullptr) {
    const long n = 2L * a.batch * (kTaps - 1) * (a.Hkv * kHeadDim / 4);
    long blocks = (n + kPrologueThreads - 1) / kPrologueThreads;
    if (blocks > 4096) blocks = 4096;
    if (blocks > 0) {
      relattn_prologue_state_kernel<<<(unsigned)blocks, kPrologueThreads, 0, stream>>>(a);
      return cudaGetLastError();
    }
  }
  return cudaSuccess;
}

}  // namespace relattn
