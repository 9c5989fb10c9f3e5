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
// once.  The main kernel is persistent and warp-specialised: a CTA walks
// tiles of T consecutive chunk tokens (about 40 KB of q, k and v); a producer
// warp streams each tile's q, k and v slabs (plus the 3 k / v rows before the
// tile, the conv halo) into a 2-stage shared-memory ring with bulk async
// copies tracked by full / empty mbarriers, and 8 consumer warps compute the
// rows from shared memory, a half-warp per 128-dim row (8 dims a lane,
// 16-byte accesses), storing straight from registers.  The conv taps sit in
// shared memory, tap-major.  Every wait is bounded; a timeout sets the device
// error word and the CTA drains its own copies before it exits.  The same
// launch writes the conv state after its tiles.
//
// The register-only kernel (one warp per 4 rows, every tap read from global
// memory) and the separate state kernel serve head counts whose tile does
// not fit in shared memory.
#include "launch.h"
#include "mxfp8.cuh"
#include "tc_common.cuh"

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
  // MXFP8 cache (null: none): E4M3 codes [total_k, Hkv, 128] and E8M0 scales
  // [total_k, Hkv, 4] of the bf16-rounded k / v rows, written beside (or
  // instead of, when k_cache / v_cache are null) the bf16 cache
  uint8_t *k8, *v8, *ks8, *vs8;
  int *err;
  int skip_tile;   // test hook: a token tile whose copies are never issued (-1: none)
};

// MXFP8 of a cache row's 32-dim block spread over 32 / N lanes (N values
// each, consecutive lanes holding consecutive dims; `mask` covers them):
// the values are rounded to bf16 first (the bf16 cache's values), the block
// max taken across the lanes.  c[i]: this lane's codes 4i .. 4i+3.
template <int N>
__device__ __forceinline__ void mx_quant_lanes(const float (&y)[N], unsigned mask, uint32_t (&c)[N / 4], int &e) {
  float v[N];
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    v[i] = __bfloat162float(__float2bfloat16_rn(y[i]));
    am = fmaxf(am, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 1; o < 32 / N; o <<= 1) am = fmaxf(am, __shfl_xor_sync(mask, am, o));
  e = mx_block_exponent(am);
  const float inv = pow2i(-e);
#pragma unroll
  for (int i = 0; i < N / 4; ++i)
    c[i] = e4m3x2(v[4 * i + 1] * inv, v[4 * i] * inv) | (e4m3x2(v[4 * i + 3] * inv, v[4 * i + 2] * inv) << 16);
}

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
      __nv_bfloat16 *cache = kind[j] == 1 ? a.k_cache : a.v_cache;
      if (kind[j] == 0) {
        store4(a.q_out + ((size_t)out_row[j] * a.Hq + head[j]) * kHeadDim + dim, y);
      } else {
        const size_t crow = (size_t)out_row[j] * a.Hkv + head[j];
        if (cache != nullptr) store4(cache + crow * kHeadDim + dim, y);
        uint8_t *codes = kind[j] == 1 ? a.k8 : a.v8;
        if (codes != nullptr) {   // (warp-uniform)
          uint32_t c[1];
          int e;
          mx_quant_lanes<4>(y, 0xffffffffu, c, e);
          *reinterpret_cast<uint32_t *>(codes + crow * kHeadDim + dim) = c[0];
          if ((lane & 7) == 0) (kind[j] == 1 ? a.ks8 : a.vs8)[crow * 4 + (lane >> 3)] = (uint8_t)(e + 127);
        }
      }
    }
  }
}

// conv state after the chunk: the last 3 pre-convolution inputs of each
// sequence (from the chunk, else from the state before it, else zero); raw
// bf16 copies, 8 bytes a thread, over [first, ...) with the given stride
__device__ __forceinline__ void state_out_pass(const PrologueArgs &a, long first, long stride) {
  const int C4 = a.Hkv * kHeadDim / 4;
  const long n = (long)a.batch * (kTaps - 1) * C4;
  for (long e = first; e < 2 * n; e += stride) {
    const bool is_k = e < n;
    const long f = is_k ? e : e - n;
    const int c4 = (int)(f % C4), jb = (int)(f / C4);
    const int j = jb % (kTaps - 1), b = jb / (kTaps - 1);
    __nv_bfloat16 *dst = is_k ? a.state_out_k : a.state_out_v;
    if (dst == nullptr) continue;
    const int cq = a.cu_q[b], Lq = a.cu_q[b + 1] - cq;
    if (cq < 0 || Lq < 0 || a.cu_q[b + 1] > a.total_q) {
      atomicOr(a.err, kDevErrSeqlens);
      continue;
    }
    const int p = Lq - (kTaps - 1) + j;                   // chunk row of state slot j
    const __nv_bfloat16 *src = is_k ? a.k : a.v;
    const __nv_bfloat16 *st = is_k ? a.state_in_k : a.state_in_v;
    uint2 u = make_uint2(0u, 0u);
    if (p >= 0) u = *reinterpret_cast<const uint2 *>(src + (size_t)(cq + p) * 4 * C4 + 4 * c4);
    else if (st != nullptr)
      u = *reinterpret_cast<const uint2 *>(st + ((size_t)b * (kTaps - 1) + (kTaps - 1 + p)) * 4 * C4 + 4 * c4);
    *reinterpret_cast<uint2 *>(dst + ((size_t)b * (kTaps - 1) + j) * 4 * C4 + 4 * c4) = u;
  }
}

__global__ void __launch_bounds__(kPrologueThreads)
relattn_prologue_state_kernel(const PrologueArgs a) {
  state_out_pass(a, (long)blockIdx.x * blockDim.x + threadIdx.x, (long)gridDim.x * blockDim.x);
}

// ------------------------------------------------------------------ staged kernel

constexpr int kConsumerWarps = 8;         // the row math
constexpr int kStagedThreads = 32 * (kConsumerWarps + 1);   // + the producer warp
constexpr int kStages = 2;
constexpr int kHalo = kTaps - 1;          // k / v rows before a tile that its taps read
constexpr int kMaxTileTokens = 32;        // (the producer warp's lanes fill the token info)
// shared memory: full / empty mbarriers, the abort flag, per-stage token info,
// the conv taps, then the stages
constexpr uint32_t kFullBarOffset = 0, kEmptyBarOffset = 64, kAbortOffset = 128;
constexpr uint32_t kInfoOffset = 256;
constexpr uint32_t kWeightOffset = (kInfoOffset + kStages * kMaxTileTokens * 16 + 127) / 128 * 128;
constexpr uint32_t kTargetStageBytes = 40u << 10;
constexpr size_t kPrologueMaxSmem = 227u << 10;
static_assert(kStages <= 8, "barrier slots");

// global -> shared bulk copy completing on an mbarrier (16-byte aligned
// addresses, a multiple of 16 bytes)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Bounded wait on an mbarrier phase that suspends the thread between probes
// (the consumer warps wait here for most of a stage's copy, and a suspended
// warp leaves the issue slots to the others).  Gives up after about a second
// of SM clocks or when another thread raised *abort, setting *abort = site.
__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                           int site) {
  const long long t0 = clock64();
  for (;;) {
    if (tc::mbar_try_wait(bar, parity, 100000u)) return true;
    if (*abort) return false;
    if (clock64() - t0 > 2000000000ll) {
      *abort = site;
      return false;
    }
  }
}

__device__ __forceinline__ void unpack8(const uint4 u, float (&x)[8]) {
  x[0] = __uint_as_float(u.x << 16);
  x[1] = __uint_as_float(u.x & 0xffff0000u);
  x[2] = __uint_as_float(u.y << 16);
  x[3] = __uint_as_float(u.y & 0xffff0000u);
  x[4] = __uint_as_float(u.z << 16);
  x[5] = __uint_as_float(u.z & 0xffff0000u);
  x[6] = __uint_as_float(u.w << 16);
  x[7] = __uint_as_float(u.w & 0xffff0000u);
}

__device__ __forceinline__ uint4 pack8(const float (&y)[8]) {
  uint4 u;
  u.x = pack_bf16x2(y[0], y[1]);
  u.y = pack_bf16x2(y[2], y[3]);
  u.z = pack_bf16x2(y[4], y[5]);
  u.w = pack_bf16x2(y[6], y[7]);
  return u;
}

// y *= g / rms(y) over one 128-dim row held by a half-warp (8 dims a lane)
__device__ __forceinline__ void rms_norm_half(float (&y)[8], const float (&g)[8], float eps,
                                              unsigned hmask) {
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(y[i], y[i], ss);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(hmask, ss, o);
  const float inv = rsqrtf(ss * (1.f / kHeadDim) + eps);
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] *= inv * g[i];
}

// Two rows at once, one per register set (their reductions interleave):
// y *= g / rms(y) for each.
__device__ __forceinline__ void rms_norm_half2(float (&y0)[8], float (&y1)[8], const float (&g)[8],
                                               float eps, unsigned hmask) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    s0 = fmaf(y0[i], y0[i], s0);
    s1 = fmaf(y1[i], y1[i], s1);
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    s0 += __shfl_xor_sync(hmask, s0, o);
    s1 += __shfl_xor_sync(hmask, s1, o);
  }
  const float inv0 = rsqrtf(s0 * (1.f / kHeadDim) + eps);
  const float inv1 = rsqrtf(s1 * (1.f / kHeadDim) + eps);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    y0[i] *= inv0 * g[i];
    y1[i] *= inv1 * g[i];
  }
}

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!tc::mbar_test_wait(bar, parity))
    if (clock64() - t0 > 200000000ll) return false;
  return true;
}

// One k / v row of a tile, loaded: the 4 conv inputs of the lane's 8 dims.
struct KvRow {
  float x[kTaps][8];
  const float *w;           // the lane's taps in shared memory: w[d * C + i], dims i < 8
  size_t crow;              // the cache row (row * Hkv + head)
  bool is_k, live;
};

// Warp-specialised: the producer warp walks the CTA's tiles (tile n in stage
// n % kStages), fills the stage's token info and issues the tile's bulk
// copies once the 8 consumer warps have released the stage; each consumer
// warp waits for the stage, does its share of the rows and releases it.  No
// block-wide barrier inside the loop.  Stage layout: q [T][Hq][128], then k
// and v [T + 3][Hkv][128] each (row j of k / v is token t0 - 3 + j).  Token
// info: {row in the sequence's chunk, cache row - token, ok, sequence}.
__global__ void __launch_bounds__(kStagedThreads, 2)
relattn_prologue_staged_kernel(const PrologueArgs a, int T) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kAbortOffset);
  int4 *info_all = reinterpret_cast<int4 *>(smem + kInfoOffset);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hq = a.Hq, Hkv = a.Hkv;
  constexpr uint32_t kRow = kHeadDim * 2;   // bytes of a row
  const uint32_t q_region = (uint32_t)T * Hq * kRow;
  const uint32_t kv_region = (uint32_t)(T + kHalo) * Hkv * kRow;
  const uint32_t stage_bytes = q_region + 2 * kv_region;
  const int C = Hkv * kHeadDim;
  const uint32_t stage0 = kWeightOffset + 2u * kTaps * C * 4;
  const int tiles = (a.total_q + T - 1) / T;
  auto full = [&](int st) { return sbase + kFullBarOffset + 8u * st; };
  auto empty = [&](int st) { return sbase + kEmptyBarOffset + 8u * st; };

  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      tc::mbar_init(full(st), 1);
      tc::mbar_init(empty(st), kConsumerWarps);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  // conv taps, transposed to tap-major so a half-warp reads 512 contiguous bytes a tap
  float *wsm = reinterpret_cast<float *>(smem + kWeightOffset);
  for (int e = tid; e < 2 * C; e += kStagedThreads) {
    const int kind = e >= C, c = e - kind * C;
    const float4 w = __ldg(reinterpret_cast<const float4 *>((kind ? a.conv_v : a.conv_k) + (size_t)c * kTaps));
    float *dst = wsm + (size_t)kind * kTaps * C + c;
    dst[0] = w.x;
    dst[C] = w.y;
    dst[2 * C] = w.z;
    dst[3 * C] = w.w;
  }
  __syncthreads();

  int issued = 0;                   // (producer) tiles whose copies were issued
  if (warp == kConsumerWarps) {
    // ======================================================== producer warp
    for (int n = 0;; ++n) {
      const int tile = (int)blockIdx.x + n * (int)gridDim.x;
      if (tile >= tiles) break;
      const int st = n % kStages;
      if (n >= kStages) {           // the consumers released tile n - kStages
        bool ok = true;
        if (lane == 0) ok = stage_wait(empty(st), ((n / kStages) - 1) & 1, abort_flag, 2);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      const int t0 = tile * T, nt = min(T, a.total_q - t0);
      if (lane < nt) {
        const int t = t0 + lane;
        const int b = seq_of(a.cu_q, a.batch, t);
        const int cq = a.cu_q[b], ck = a.cu_k[b];
        const int Lq = a.cu_q[b + 1] - cq, Lk = a.cu_k[b + 1] - ck;
        const int pos = t - cq;
        const bool ok = pos >= 0 && pos < Lq && Lk >= Lq && ck >= 0 && a.cu_k[b + 1] <= a.total_k;
        if (!ok) atomicOr(a.err, kDevErrSeqlens);
        info_all[st * kMaxTileTokens + lane] = make_int4(pos, ck + (Lk - Lq) - cq, ok ? 1 : 0, b);
      }
      __syncwarp();
      if (lane == 0 && tile != a.skip_tile) {
        const int t1 = t0 + nt, h0 = max(0, t0 - kHalo);
        const uint32_t qb = (uint32_t)nt * Hq * kRow;
        const uint32_t kvb = (uint32_t)(t1 - h0) * Hkv * kRow;
        const uint32_t kv_dst = (uint32_t)(h0 - (t0 - kHalo)) * Hkv * kRow;
        const uint32_t dst = sbase + stage0 + (uint32_t)st * stage_bytes;
        tc::mbar_arrive_expect_tx(full(st), qb + 2 * kvb);
        bulk_load(dst, a.q + (size_t)t0 * Hq * kHeadDim, qb, full(st));
        bulk_load(dst + q_region + kv_dst, a.k + (size_t)h0 * Hkv * kHeadDim, kvb, full(st));
        bulk_load(dst + q_region + kv_region + kv_dst, a.v + (size_t)h0 * Hkv * kHeadDim, kvb,
                  full(st));
      }
      ++issued;
    }
  } else {
    // ======================================================== consumer warps
    // a half-warp takes a row, lane hl of it dims 8hl .. 8hl+7
    const int hw = tid >> 4, hl = tid & 15, dim = 8 * hl;
    const unsigned hmask = 0xffffu << (lane & 16);
    constexpr int kHalves = 2 * kConsumerWarps;
    float gq[8], gk[8];
    {
      const float4 *pq = reinterpret_cast<const float4 *>(a.norm_q + dim);
      const float4 *pk = reinterpret_cast<const float4 *>(a.norm_k + dim);
      const float4 q0 = __ldg(pq), q1 = __ldg(pq + 1), k0 = __ldg(pk), k1 = __ldg(pk + 1);
      gq[0] = q0.x; gq[1] = q0.y; gq[2] = q0.z; gq[3] = q0.w;
      gq[4] = q1.x; gq[5] = q1.y; gq[6] = q1.z; gq[7] = q1.w;
      gk[0] = k0.x; gk[1] = k0.y; gk[2] = k0.z; gk[3] = k0.w;
      gk[4] = k1.x; gk[5] = k1.y; gk[6] = k1.z; gk[7] = k1.w;
    }
    int n = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++n) {
      const int st = n % kStages;
      const bool ok = stage_wait(full(st), (n / kStages) & 1, abort_flag, 1);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int t0 = tile * T, nt = min(T, a.total_q - t0);
      const uint8_t *sq = smem + stage0 + (size_t)st * stage_bytes;
      const uint8_t *skv = sq + q_region;
      const int4 *info = info_all + st * kMaxTileTokens;

      // ---- q rows: the tile's q slab is the rows t0*Hq .. (t0+nt)*Hq of q;
      // two rows per half-warp and pass (the second re-reads the first's row
      // when it is past the end, and is not stored)
      const int q_rows = nt * Hq;
      for (int r0 = hw; r0 < q_rows; r0 += 2 * kHalves) {
        const int r1 = r0 + kHalves;
        const bool two = r1 < q_rows;
        float y0[8], y1[8];
        unpack8(*reinterpret_cast<const uint4 *>(sq + (size_t)r0 * kRow + 16 * hl), y0);
        unpack8(*reinterpret_cast<const uint4 *>(sq + (size_t)(two ? r1 : r0) * kRow + 16 * hl), y1);
        rms_norm_half2(y0, y1, gq, a.eps, hmask);
        __nv_bfloat16 *o = a.q_out + (size_t)t0 * Hq * kHeadDim + dim;
        *reinterpret_cast<uint4 *>(o + (size_t)r0 * kHeadDim) = pack8(y0);
        if (two) *reinterpret_cast<uint4 *>(o + (size_t)r1 * kHeadDim) = pack8(y1);
      }

      // ---- k / v rows, order (token, k heads, v heads)
      const int kv_rows = nt * 2 * Hkv;
      auto load_kv = [&](int r, KvRow &R) {
        const int tt = r / (2 * Hkv), rem = r - tt * 2 * Hkv;
        R.is_k = rem < Hkv;
        const int h = R.is_k ? rem : rem - Hkv;
        const int4 in = info[tt];
        R.live = in.z != 0;
        const int pos = in.x;
        // row tt + 3 - d of the stage's k (or v) block is token t - d
        const uint8_t *src = skv + (R.is_k ? 0u : kv_region) + ((size_t)(tt + kHalo) * Hkv + h) * kRow + 16 * hl;
#pragma unroll
        for (int d = 0; d < kTaps; ++d)
          unpack8(*reinterpret_cast<const uint4 *>(src - (size_t)d * Hkv * kRow), R.x[d]);
        if (R.live && pos < kHalo) {
          // taps before the chunk: the conv state, or zero (the stage rows
          // there belong to another sequence, or were never loaded)
          const __nv_bfloat16 *state = R.is_k ? a.state_in_k : a.state_in_v;
#pragma unroll
          for (int d = 1; d < kTaps; ++d) {
            if (pos - d >= 0) continue;
            if (state != nullptr) {
              unpack8(*reinterpret_cast<const uint4 *>(
                          state + ((size_t)in.w * kHalo + (kHalo + pos - d)) * Hkv * kHeadDim +
                          (size_t)h * kHeadDim + dim),
                      R.x[d]);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) R.x[d][i] = 0.f;
            }
          }
        }
        R.w = wsm + (R.is_k ? 0 : kTaps * C) + h * kHeadDim + dim;
        R.crow = (size_t)(t0 + tt + in.y) * Hkv + h;
      };
      auto conv = [&](const KvRow &R, float (&y)[8]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = R.x[0][i];   // the input added back
#pragma unroll
        for (int d = 0; d < kTaps; ++d) {
          const float4 w0 = *reinterpret_cast<const float4 *>(R.w + d * C);
          const float4 w1 = *reinterpret_cast<const float4 *>(R.w + d * C + 4);
          const float wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) y[i] = fmaf(wd[i], R.x[d][i], y[i]);
        }
      };
      for (int r = hw; r < kv_rows; r += kHalves) {
        KvRow A;
        load_kv(r, A);
        float y[8];
        conv(A, y);
        if (A.is_k) rms_norm_half(y, gk, a.eps, hmask);
        __nv_bfloat16 *cache = A.is_k ? a.k_cache : a.v_cache;
        if (A.live && cache != nullptr) *reinterpret_cast<uint4 *>(cache + A.crow * kHeadDim + dim) = pack8(y);
        uint8_t *codes = A.is_k ? a.k8 : a.v8;
        if (codes != nullptr) {   // (uniform over the half-warp: one row)
          uint32_t c[2];
          int e;
          mx_quant_lanes<8>(y, hmask, c, e);
          if (A.live) {
            *reinterpret_cast<uint2 *>(codes + A.crow * kHeadDim + dim) = make_uint2(c[0], c[1]);
            if ((hl & 3) == 0) (A.is_k ? a.ks8 : a.vs8)[A.crow * 4 + (hl >> 2)] = (uint8_t)(e + 127);
          }
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty(st));   // this warp is done with the stage
    }
  }
  __syncthreads();
  if (*abort_flag) {
    if (warp == kConsumerWarps && lane == 0) {
      record_timeout(a.err, *abort_flag);
      // copies still in flight: those of the last kStages tiles issued
      for (int m = max(0, issued - kStages); m < issued; ++m)
        drain_wait(full(m % kStages), (m / kStages) & 1);
    }
    return;
  }
  // the conv state after the chunk, spread over the grid
  if (a.state_out_k != nullptr || a.state_out_v != nullptr)
    state_out_pass(a, (long)blockIdx.x * blockDim.x + tid, (long)gridDim.x * blockDim.x);
}

}  // namespace

cudaError_t launch_prologue(const relattn_prologue_params *p, int *err, int sms, int skip_tile,
                            cudaStream_t stream, const relattn_kv_mxfp8_out *mx) {
  PrologueArgs a;
  a.skip_tile = skip_tile;
  a.k8 = mx ? static_cast<uint8_t *>(mx->k) : nullptr;
  a.v8 = mx ? static_cast<uint8_t *>(mx->v) : nullptr;
  a.ks8 = mx ? static_cast<uint8_t *>(mx->k_scale) : nullptr;
  a.vs8 = mx ? static_cast<uint8_t *>(mx->v_scale) : nullptr;
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
  // staged kernel: tokens per tile so that a stage holds about kTargetStageBytes
  const uint32_t tok_bytes = (uint32_t)(a.Hq + 2 * a.Hkv) * kHeadDim * 2;
  int T = (int)(kTargetStageBytes / tok_bytes);
  T = T < 1 ? 1 : (T > kMaxTileTokens ? kMaxTileTokens : T);
  const size_t stage_bytes = (size_t)T * a.Hq * kHeadDim * 2 + 2 * (size_t)(T + kHalo) * a.Hkv * kHeadDim * 2;
  const size_t smem = kWeightOffset + 2 * kTaps * (size_t)a.Hkv * kHeadDim * 4 + kStages * stage_bytes;
  if (rows > 0 && smem <= kPrologueMaxSmem) {
    static std::atomic<bool> attr_set[kMaxDevicesAttr];   // the attribute is set once per device
    cudaError_t e = set_max_smem_once(reinterpret_cast<const void *>(relattn_prologue_staged_kernel),
                                      (int)kPrologueMaxSmem, attr_set);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, relattn_prologue_staged_kernel, kStagedThreads, smem);
    if (e != cudaSuccess) return e;
    const long tiles = (a.total_q + T - 1) / T;
    long grid = (long)(sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
    if (grid > tiles) grid = tiles;
    relattn_prologue_staged_kernel<<<(unsigned)grid, kStagedThreads, smem, stream>>>(a, T);
    return cudaGetLastError();   // (it also writes the conv state)
  }
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
