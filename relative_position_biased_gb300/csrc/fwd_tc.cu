// fwd_tc.cu -- relative-attention prefill on 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory, TMA-fed K/V).
//
// Same computation as the definition on the page "SGLang and Miles Add Day-0
// Support for Inkling", section "Attention with Relative Positional
// Embedding":  x(i,j) = s(i) * (alpha q_i.k_j + [0 <= i-j < E] r_i . P[:, i-j]),
// online softmax, PV.
//
// One CTA = one query head x 128 query rows (TMEM lane a <-> row a), keys in
// tiles of 64, visited from the diagonal backwards.  Warp roles:
//   warp 0      TMA producer for K and V tiles (4-stage ring)
//   warp 1      MMA issuer (one thread):  S = Q K^T (Q in TMEM),
//               R_chunk = r P[:, 64c..64c+64) (both operands from shared
//               memory), O += P V (P in TMEM)
//   warp 2      TMEM allocator; producer of the P slices (plain loads into
//               the 128-byte-swizzled layout)
//   warps 4-11  softmax, two warpgroups: row a is owned by one thread of each
//               (TMEM lane a); warpgroup wg takes keys [32 wg, 32 wg + 32) of
//               every tile.  They write the q / r rows, load S from TMEM, add
//               the relative bias, mask edge tiles, agree on the running row
//               max through shared memory, write P (bf16) back over S, rescale
//               their half of O when the max grows by more than 2^8, and write
//               out / lse at the end.
//
// Tensor memory (512 columns): Q [0,64) bf16, S0 [64,128), S1 [128,192),
// O [192,320), R ring [320,512) = three 64-distance chunks of r.P.
//
// Relative bias without a sheared tensor: the R ring holds, for every row, the
// relative logits of three consecutive 64-distance chunks.  Key tile at
// offset D = i_0 - j_0 needs distances D-63 .. D+127 (chunks D/64-1 .. D/64+1);
// walking tiles away from the diagonal needs one new chunk per tile.  Each
// thread loads a 64-column window of its own row (one load shape for the
// whole warp) and shifts it by its lane index with a 5-stage select network,
// which turns "distance order" into "key order" in registers.
//
// Every wait is bounded; a timeout sets the device error word, the CTA drains
// its own copies / MMAs with bounded waits, frees TMEM and exits.
#include <cudaTypedefs.h>

#include "launch.h"
#include "tc_common.cuh"

namespace relattn {
namespace {

using namespace tc;

constexpr int BM = 128;          // query rows per CTA
constexpr int BN = 64;           // keys per tile
constexpr int KV_STAGES = 4;
constexpr int P_STAGES = 4;
constexpr int NTHREADS = 384;
constexpr float kRescaleThreshold = 8.f;   // log2 units

// TMEM columns
constexpr uint32_t TM_Q = 0, TM_S0 = 64, TM_O = 192, TM_R = 320;

// Shared memory layout (offsets from a 1024-aligned base)
constexpr uint32_t SM_KV = 0;                                  // stages of K(16K) + V(16K)
constexpr uint32_t KV_STAGE_BYTES = 32768;
constexpr uint32_t SM_RT = SM_KV + KV_STAGES * KV_STAGE_BYTES;  // r tile 16K
constexpr uint32_t SM_PS = SM_RT + 16384;                      // P slices 2 x 8K
constexpr uint32_t SM_BAR = SM_PS + P_STAGES * 8192;
// barriers (8 bytes each)
constexpr int B_KV_FULL = 0, B_KV_EMPTY = B_KV_FULL + KV_STAGES, B_PS_FULL = B_KV_EMPTY + KV_STAGES,
              B_PS_EMPTY = B_PS_FULL + P_STAGES, B_RT_FULL = B_PS_EMPTY + P_STAGES,
              B_Q_READY = B_RT_FULL + 1, B_S_FULL = B_Q_READY + 1, B_P_FULL = B_S_FULL + 2,
              B_PV_DONE = B_P_FULL + 2, B_R_FULL = B_PV_DONE + 2, B_R_FREE = B_R_FULL + 3,
              B_DRAIN = B_R_FREE + 1, B_XCH = B_DRAIN + 1, B_COUNT = B_XCH + 4;
constexpr uint32_t SM_TMEM_SLOT = SM_BAR + B_COUNT * 8;
constexpr uint32_t SM_ABORT = SM_TMEM_SLOT + 8;
constexpr uint32_t SM_XCH = SM_ABORT + 8;                      // row-max exchange [2][2][128] f32
constexpr uint32_t SM_TOTAL = SM_XCH + 2 * 2 * 128 * 4;
constexpr uint32_t SMEM_BYTES = SM_TOTAL + 1024;  // + alignment slack

struct TcArgs {
  KernelArgs a;
  int has_bias;
};

__device__ __forceinline__ int floor_div64(int x) { return x >= 0 ? x >> 6 : -((63 - x) >> 6); }

template <bool DECODE>
__global__ void __launch_bounds__(NTHREADS, 1)
relattn_fwd_tc_kernel(const __grid_constant__ TcArgs ta,
                              const __grid_constant__ CUtensorMap map_k,
                              const __grid_constant__ CUtensorMap map_v) {
  const KernelArgs &a = ta.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sb = smem_addr(smem);
  auto bar = [&](int i) { return sb + SM_BAR + 8u * i; };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM_ABORT);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ------------------------------------------------------------ work item
  // prefill: one query head x 128 consecutive rows.  decode: 128 rows of the
  // (token, head-in-group) list of one kv head, and one split of its keys.
  int b, kv_head, row0, nrows, split = 0, h_fixed = 0;
  if constexpr (DECODE) {
    split = blockIdx.x;
    kv_head = blockIdx.y / a.row_blocks;
    row0 = (blockIdx.y % a.row_blocks) * BM;
    b = blockIdx.z;
  } else {
    h_fixed = blockIdx.y;
    kv_head = h_fixed / a.group;
    row0 = (a.q_tiles - 1 - blockIdx.x) * BM;   // longest-running tiles first
    b = blockIdx.z;
  }
  const int cq = a.cu_q[b], ck = a.cu_k[b];
  const int Lq = a.cu_q[b + 1] - cq, Lk = a.cu_k[b + 1] - ck;
  if (Lq < 0 || Lk < Lq || Lq > a.max_q || Lk > a.max_k) {
    if (tid == 0) atomicOr(a.err, kDevErrSeqlens);
    return;
  }
  nrows = min(BM, (DECODE ? Lq * a.group : Lq) - row0);
  if (nrows <= 0) return;
  const int off = Lk - Lq;
  // row (local, clamped to the last valid one) -> token t and query head
  auto row_t = [&](int rl) {
    const int x = row0 + min(rl, nrows - 1);
    return DECODE ? x / a.group : x;
  };
  auto row_h = [&](int rl) {
    const int x = row0 + min(rl, nrows - 1);
    return DECODE ? kv_head * a.group + x % a.group : h_fixed;
  };
  const int p0 = off + row_t(0), p_last = off + row_t(nrows - 1);
  const int j_lo = a.window > 0 ? max(0, p0 - a.window + 1) : 0;
  // distance offset D(n) = p0 - j0(n) of the key tile processed n-th (from the
  // diagonal backwards); rows sit at p0 + delta, delta <= span
  int ntiles, D_first, span;
  if constexpr (DECODE) {
    const int kbase = j_lo & ~(BN - 1);
    const int kbeg = kbase + split * a.split_chunk;
    const int kend = min(p_last + 1, kbeg + a.split_chunk);
    ntiles = kend > kbeg ? (kend - kbeg + BN - 1) / BN : 0;
    D_first = p0 - (kbeg + (ntiles - 1) * BN);
    span = p_last - p0;
  } else {
    // key tiles start at j0(n) = p0 + 64 - 64 n  (D = 64 n - 64), or one tile
    // later when every row of the block sits in the first 64 positions
    D_first = (p_last >= p0 + BN) ? -BN : 0;
    ntiles = (p0 - j_lo - D_first + BN - 1) / BN + 1;
    span = BM - 1;   // padding rows reuse the pattern of full tiles
  }
  auto tile_D = [&](int n) { return D_first + BN * n; };
  // band tiles (some distance < E) form a prefix of the tile order
  int nband = 0;
  if (ta.has_bias && ntiles > 0) {
    const int lim = a.E + BN - 1;  // band iff D - 63 < E
    nband = tile_D(ntiles - 1) < lim ? ntiles : max(0, (lim - D_first + BN - 1) / BN);
    if (nband > ntiles) nband = ntiles;
  }
  // newest 64-distance chunk of r.P a tile needs (one more per tile)
  auto c_new = [&](int n) { return floor_div64(tile_D(n) + span); };
  const int c_first = c_new(0);
  const int c_last = nband > 0 ? c_new(nband - 1) : -1;
  // first chunk computed: the oldest one tile 0 reads (a decode split far from
  // the diagonal starts deep in the band).  Chunk c uses ring slot / P stage /
  // barrier phase counted from c_start.
  const int c_start = nband > 0 ? max(0, floor_div64(tile_D(0) - (BN - 1))) : 0;

  // ------------------------------------------------------------ setup
  if (tid == 0) {
    for (int i = 0; i < KV_STAGES; ++i) {
      mbar_init(bar(B_KV_FULL + i), 1);
      mbar_init(bar(B_KV_EMPTY + i), 1);
    }
    for (int i = 0; i < P_STAGES; ++i) {
      mbar_init(bar(B_PS_FULL + i), 1);
      mbar_init(bar(B_PS_EMPTY + i), 1);
    }
    mbar_init(bar(B_RT_FULL), 256);
    mbar_init(bar(B_Q_READY), 256);
    mbar_init(bar(B_S_FULL + 0), 1);
    mbar_init(bar(B_S_FULL + 1), 1);
    mbar_init(bar(B_P_FULL + 0), 256);
    mbar_init(bar(B_P_FULL + 1), 256);
    mbar_init(bar(B_PV_DONE + 0), 1);
    mbar_init(bar(B_PV_DONE + 1), 1);
    for (int i = 0; i < 3; ++i) mbar_init(bar(B_R_FULL + i), 1);
    mbar_init(bar(B_R_FREE), 256);
    mbar_init(bar(B_DRAIN), 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar(B_XCH + i), 64);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(sb + SM_TMEM_SLOT, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map_k);
    prefetch_tmap(&map_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + SM_TMEM_SLOT);

  if (warp == 0) {
    // ======================================================== K/V producer
    if (lane == 0) {
      int issued = 0;
      for (int n = 0; n < ntiles && !*abort_flag; ++n) {
        const int st = n % KV_STAGES;
        if (n >= KV_STAGES && !mbar_wait(bar(B_KV_EMPTY + st), ((n / KV_STAGES) - 1) & 1, abort_flag, 1))
          break;
        const int key = ck + p0 - tile_D(n);   // may be < 0: the tile reads zeros there
        const uint32_t dst = sb + SM_KV + st * KV_STAGE_BYTES;
        mbar_arrive_expect_tx(bar(B_KV_FULL + st), KV_STAGE_BYTES);
        tma_load_3d(dst, &map_k, 0, kv_head, key, bar(B_KV_FULL + st));
        tma_load_3d(dst + 8192, &map_k, 64, kv_head, key, bar(B_KV_FULL + st));
        tma_load_3d(dst + 16384, &map_v, 0, kv_head, key, bar(B_KV_FULL + st));
        tma_load_3d(dst + 24576, &map_v, 64, kv_head, key, bar(B_KV_FULL + st));
        issued = n + 1;
      }
      if (*abort_flag) {
        // let our own copies land before the CTA goes away (bounded, not cut short by the abort)
        volatile int keep_waiting = 0;
        for (int n = max(0, issued - KV_STAGES); n < issued; ++n)
          mbar_wait(bar(B_KV_FULL + n % KV_STAGES), (n / KV_STAGES) & 1, &keep_waiting, 2, 400000000ll);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ======================================================== P-slice producer
    // Chunk c = P[:, 64c, 64c+64) as rd_pad rows (channels) of 128 bytes in the
    // 128-byte-swizzled layout the MMA descriptor expects; zero outside [0, E)
    // and past r_dim.  Plain 16-byte loads (P is small and L2-resident).
    if (nband > 0) {
      const int c_hi = min(c_last, (a.E - 1) / BN);     // chunks past E stay zero-filled
      for (int c = c_start; c <= c_last; ++c) {
        const int o = c - c_start;
        const int st = o % P_STAGES;
        if (o >= P_STAGES) {
          const bool w = mbar_wait(bar(B_PS_EMPTY + st), ((o / P_STAGES) - 1) & 1, abort_flag, 3);
          if (!__all_sync(0xffffffffu, w)) break;
        }
        uint8_t *dst = smem + SM_PS + st * 8192;
        // up to 64 channels x 8 sixteen-byte pieces = 16 per lane: issue every
        // load before the first store so the L2 round trips overlap
        uint4 v[16];
#pragma unroll
        for (int it = 0; it < 16; ++it) {
          const int idx = lane + 32 * it, ch = idx >> 3, j = idx & 7, col = BN * c + 8 * j;
          v[it] = make_uint4(0u, 0u, 0u, 0u);
          if (idx < a.rd_pad * 8 && c <= c_hi && ch < a.rd && col < a.E)
            v[it] = *reinterpret_cast<const uint4 *>(a.P + (size_t)ch * a.E + col);
        }
#pragma unroll
        for (int it = 0; it < 16; ++it) {
          const int idx = lane + 32 * it, ch = idx >> 3, j = idx & 7;
          if (idx < a.rd_pad * 8)
            *reinterpret_cast<uint4 *>(dst + (ch >> 3) * 1024 + (ch & 7) * 128 +
                                       ((j ^ (ch & 7)) << 4)) = v[it];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PS_FULL + st));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================================================== MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(BM, BN, 0, 0);       // S: Q(tmem) x K(smem, K-major)
      const uint32_t id_o = idesc_bf16_f32(BM, 128, 0, 1);      // O: P(tmem) x V(smem, MN-major)
      const uint32_t id_r = idesc_bf16_f32(BM, BN, 0, 1);       // R: r(smem) x P(smem, MN-major)
      const int r_ksteps = a.rd_pad / 16;
      // descriptor bases; per k-step / stage only the 16-byte address field moves
      const uint64_t kd0 = smem_desc_sw128(sb + SM_KV, 16, 1024);
      const uint64_t vd0 = smem_desc_sw128(sb + SM_KV + 16384, 8192, 1024);
      const uint64_t rd0 = smem_desc_sw128(sb + SM_RT, 16, 1024);
      const uint64_t pd0 = smem_desc_sw128(sb + SM_PS, 8192, 1024);
      bool ok = mbar_wait(bar(B_Q_READY), 0, abort_flag, 6);
      tc_fence_after();
      bool rt_ready = false;
      auto issue_r = [&](int c) -> bool {
        if (!rt_ready) {
          if (!mbar_wait(bar(B_RT_FULL), 0, abort_flag, 7)) return false;
          rt_ready = true;
        }
        const int o = c - c_start;
        const int st = o % P_STAGES;
        if (!mbar_wait(bar(B_PS_FULL + st), (o / P_STAGES) & 1, abort_flag, 8)) return false;
        tc_fence_after();
        const uint32_t d = tmem + TM_R + 64u * (uint32_t)(o % 3);
        const uint64_t pd = pd0 + (uint64_t)((st * 8192) >> 4);
        mma_ss_c<0>(d, rd0, pd, id_r);
        if (r_ksteps > 1) mma_ss_c<1>(d, rd0 + 2, pd + 128, id_r);
        if (r_ksteps > 2) mma_ss_c<1>(d, rd0 + 4, pd + 256, id_r);
        if (r_ksteps > 3) mma_ss_c<1>(d, rd0 + 6, pd + 384, id_r);
        mma_commit(bar(B_R_FULL + o % 3));
        mma_commit(bar(B_PS_EMPTY + st));
        return true;
      };
      auto issue_s = [&](int n) -> bool {
        const int st = n % KV_STAGES;
        if (!mbar_wait(bar(B_KV_FULL + st), (n / KV_STAGES) & 1, abort_flag, 9)) return false;
        tc_fence_after();
        const uint32_t d = tmem + TM_S0 + 64u * (uint32_t)(n & 1);
        const uint64_t kd = kd0 + (uint64_t)((st * KV_STAGE_BYTES) >> 4);
        const uint32_t qa = tmem + TM_Q;
        // k-step k: box k/4 (+8 KB), 32 bytes per step inside the 128-byte row
        mma_ts_c<0>(d, qa + 0, kd + 0, id_s);
        mma_ts_c<1>(d, qa + 8, kd + 2, id_s);
        mma_ts_c<1>(d, qa + 16, kd + 4, id_s);
        mma_ts_c<1>(d, qa + 24, kd + 6, id_s);
        mma_ts_c<1>(d, qa + 32, kd + 512, id_s);
        mma_ts_c<1>(d, qa + 40, kd + 514, id_s);
        mma_ts_c<1>(d, qa + 48, kd + 516, id_s);
        mma_ts_c<1>(d, qa + 56, kd + 518, id_s);
        mma_commit(bar(B_S_FULL + (n & 1)));
        return true;
      };
      if (ok && nband > 0)
        for (int c = c_start; c <= c_first && ok; ++c) ok = issue_r(c);
      if (ok && ntiles > 0) ok = issue_s(0);   // an empty decode split issues nothing
      for (int n = 0; n < ntiles && ok; ++n) {
        if (n + 1 < ntiles && !(ok = issue_s(n + 1))) break;
        if (n + 1 < nband) {
          const int c = c_new(n + 1);
          if (!(ok = mbar_wait(bar(B_R_FREE), n & 1, abort_flag, 10))) break;
          if (c >= 0 && !(ok = issue_r(c))) break;
        }
        if (!(ok = mbar_wait(bar(B_P_FULL + (n & 1)), (n >> 1) & 1, abort_flag, 11))) break;
        tc_fence_after();
        const int st = n % KV_STAGES;
        const uint64_t vd = vd0 + (uint64_t)((st * KV_STAGE_BYTES) >> 4);
        const uint32_t pa = tmem + TM_S0 + 64u * (uint32_t)(n & 1);
        // k-step k = 16 keys = 2048 bytes of the MN-major V tile
        if (n > 0) mma_ts_c<1>(tmem + TM_O, pa + 0, vd + 0, id_o);
        else mma_ts_c<0>(tmem + TM_O, pa + 0, vd + 0, id_o);
        mma_ts_c<1>(tmem + TM_O, pa + 8, vd + 128, id_o);
        mma_ts_c<1>(tmem + TM_O, pa + 16, vd + 256, id_o);
        mma_ts_c<1>(tmem + TM_O, pa + 24, vd + 384, id_o);
        mma_commit(bar(B_PV_DONE + (n & 1)));
        mma_commit(bar(B_KV_EMPTY + st));
      }
      // drain: every MMA issued above has finished before TMEM is released
      mma_commit(bar(B_DRAIN));
      volatile int keep_waiting = 0;
      mbar_wait(bar(B_DRAIN), 0, &keep_waiting, 12, 400000000ll);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ======================================================== softmax
    // Two warpgroups share the 128 rows: warpgroup wg handles keys
    // [32 wg, 32 wg + 32) of every 64-key tile (and O / output columns
    // [64 wg, 64 wg + 64)).  The two threads of a row agree on the running max
    // through a shared-memory exchange guarded by a per-lane-quarter mbarrier.
    const int wg = (warp - 4) >> 2;
    const int wq = warp & 3;                     // lane quarter (TMEM lanes 32 wq ..)
    const int a_row = 32 * wq + lane;            // row == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    const int t_row = row_t(a_row), h_row = row_h(a_row);
    // position of this row; prefill padding rows (a_row >= nrows) continue the
    // diagonal pattern and only compute garbage that is never stored
    const int pos = DECODE ? off + t_row : p0 + a_row;
    const int delta = pos - p0;                  // 0 .. span
    const int delta_w = DECODE ? off + row_t(32 * wq) - p0 : 32 * wq;   // first row of the warp
    const float sc = log_scale(min(pos, p_last), a.inv_ln_base);
    const float cqk = a.alpha_log2e * sc, cbias = kLog2e * sc;
    float *xbuf = reinterpret_cast<float *>(smem + SM_XCH);   // [2 parity][2 wg][128]

    // q row half -> TMEM columns [32 wg, 32 wg + 32) (bf16 pairs)
    {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          a.q + ((size_t)(cq + t_row) * a.Hq + h_row) * kHeadDim + 64 * wg);
      uint32_t r[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = src[i];
        r[4 * i] = v.x; r[4 * i + 1] = v.y; r[4 * i + 2] = v.z; r[4 * i + 3] = v.w;
      }
      __syncwarp();
      tmem_st32(tmem + lane_base + TM_Q + 32u * wg, r);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_Q_READY));
    }
    // r row half -> shared r tile (row a, 128-byte swizzle; zero past r_dim)
    if (nband > 0) {
      const __nv_bfloat16 *rsrc = a.r + ((size_t)(cq + t_row) * a.Hq + h_row) * a.rd;
      uint8_t *rrow = smem + SM_RT + (a_row >> 3) * 1024 + (a_row & 7) * 128;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = 4 * wg + jj;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (8 * j < a.rd) v = *reinterpret_cast<const uint4 *>(rsrc + 8 * j);
        *reinterpret_cast<uint4 *>(rrow + ((j ^ (a_row & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(B_RT_FULL));
    }

    // every lane of a softmax warp takes the same branch after a wait, so the
    // warp-collective tcgen05 loads / stores that follow see a converged warp
    auto warp_wait = [&](uint32_t br, uint32_t parity, int site) -> bool {
      const bool r = mbar_wait(br, parity, abort_flag, site);
      return __all_sync(0xffffffffu, r);
    };
    // TMEM address of distances d0 .. d0+31; valid for chunks >= c_start
    auto r_addr = [&](int d0) {
      return tmem + lane_base + TM_R + 64u * (uint32_t)(((d0 >> 6) - c_start) % 3) + (uint32_t)(d0 & 63);
    };
    const int d_min = BN * c_start;   // smaller distances were never computed (not needed)
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int n = 0; n < ntiles; ++n) {
      const uint32_t sbuf = tmem + lane_base + TM_S0 + 64u * (uint32_t)(n & 1);
      if (!(ok = warp_wait(bar(B_S_FULL + (n & 1)), (n >> 1) & 1, 13))) break;
      const int D = tile_D(n);
      const int j0 = p0 - D;
      const bool band = n < nband;
      if (band) {
        // the newest chunk this tile needs (older ones were awaited before)
        if (n == 0) {
          for (int c = c_start; c <= c_first && ok; ++c)
            ok = warp_wait(bar(B_R_FULL + (c - c_start) % 3), ((c - c_start) / 3) & 1, 14);
        } else {
          const int c = c_new(n);
          if (c >= c_start) ok = warp_wait(bar(B_R_FULL + (c - c_start) % 3), ((c - c_start) / 3) & 1, 15);
        }
        if (!ok) break;
      }
      tc_fence_after();
      uint32_t sr[32];
      __syncwarp();
      tmem_ld32(sbuf + 32u * wg, sr);
      float x[32];
      if constexpr (!DECODE) {
        // distances D + a - (32 wg + u), u in [0, 32): window [base, base + 64),
        // base a multiple of 32 (D is a multiple of 64 here)
        const int base = D + 32 * wq - 32 * wg - 32;
        uint32_t w0[32], w1[32];
        if (band) {
          if (base >= d_min) tmem_ld32(r_addr(base), w0);
          if (base + 32 >= d_min) tmem_ld32(r_addr(base + 32), w1);
        }
        tmem_wait_ld(sr);
        reg_dep(w0);
        reg_dep(w1);
        if (band) {
          // z[63 - i] = window[i]; the thread of lane t needs window[32 + t - u]
          float z[64];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            z[63 - i] = base >= d_min ? __uint_as_float(w0[i]) : 0.f;
            z[31 - i] = base + 32 >= d_min ? __uint_as_float(w1[i]) : 0.f;
          }
          tc_fence_before();
          mbar_arrive(bar(B_R_FREE));
          // y[u] = z[u + sh], sh = 31 - lane: shift with a select network
          const int sh = 31 - lane;
#pragma unroll
          for (int i = 0; i < 47; ++i) z[i] = (sh & 16) ? z[i + 16] : z[i];
#pragma unroll
          for (int i = 0; i < 39; ++i) z[i] = (sh & 8) ? z[i + 8] : z[i];
#pragma unroll
          for (int i = 0; i < 35; ++i) z[i] = (sh & 4) ? z[i + 4] : z[i];
#pragma unroll
          for (int i = 0; i < 33; ++i) z[i] = (sh & 2) ? z[i + 2] : z[i];
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] = (sh & 1) ? z[i + 1] : z[i];
#pragma unroll
          for (int u = 0; u < 32; u += 2)
            ffma2(x[u], x[u + 1], __uint_as_float(sr[u]), __uint_as_float(sr[u + 1]), cqk, cqk,
                  z[u] * cbias, z[u + 1] * cbias);
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) x[u] = __uint_as_float(sr[u]) * cqk;
        }
      } else {
        tmem_wait_ld(sr);
        if (band) {
          // rows of a warp span at most 16 positions: distances
          // D + delta - (32 wg + u) lie in a 96-wide window [bal, bal + 96)
          // starting at a multiple of 32
          const int lo = D + delta_w - 32 * wg - 31;
          const int bal = lo & ~31;
          float z[96];
#pragma unroll
          for (int hh = 0; hh < 3; ++hh) {
            uint32_t w[32];
            const int d0 = bal + 32 * hh;
            if (d0 >= d_min) {
              __syncwarp();
              tmem_ld32(r_addr(d0), w);
              tmem_wait_ld(w);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) z[95 - (32 * hh + i)] = d0 >= d_min ? __uint_as_float(w[i]) : 0.f;
          }
          tc_fence_before();
          mbar_arrive(bar(B_R_FREE));
          // y[u] = window[i0 - u] = z[95 - i0 + u] with 95 - i0 in [18, 64]
          const int i0 = D + delta - 32 * wg - bal;
          const int sh = 95 - i0 - 18;
          float* zz = z + 18;   // 78 entries
#pragma unroll
          for (int i = 0; i < 46; ++i) zz[i] = (sh & 32) ? zz[i + 32] : zz[i];
#pragma unroll
          for (int i = 0; i < 47; ++i) zz[i] = (sh & 16) ? zz[i + 16] : zz[i];
#pragma unroll
          for (int i = 0; i < 39; ++i) zz[i] = (sh & 8) ? zz[i + 8] : zz[i];
#pragma unroll
          for (int i = 0; i < 35; ++i) zz[i] = (sh & 4) ? zz[i + 4] : zz[i];
#pragma unroll
          for (int i = 0; i < 33; ++i) zz[i] = (sh & 2) ? zz[i + 2] : zz[i];
#pragma unroll
          for (int i = 0; i < 32; ++i) zz[i] = (sh & 1) ? zz[i + 1] : zz[i];
#pragma unroll
          for (int u = 0; u < 32; u += 2)
            ffma2(x[u], x[u + 1], __uint_as_float(sr[u]), __uint_as_float(sr[u + 1]), cqk, cqk,
                  zz[u] * cbias, zz[u + 1] * cbias);
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) x[u] = __uint_as_float(sr[u]) * cqk;
        }
      }
      const bool need_mask = (j0 + BN - 1 > p0) || (a.window > 0 && j0 < p_last - a.window + 1) || (j0 < 0);
      (void)delta;
      if (need_mask) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int j = j0 + 32 * wg + i;
          const bool vis = j <= pos && j >= 0 && (a.window <= 0 || pos - j < a.window);
          x[i] = vis ? x[i] : -INFINITY;
        }
      }
      float mloc = fmax3(x[0], x[1], x[2]);
#pragma unroll
      for (int i = 3; i < 31; i += 2) mloc = fmax3(mloc, x[i], x[i + 1]);
      mloc = fmaxf(mloc, x[31]);
      // agree on the row max with the other warpgroup
      float *xb = xbuf + (n & 1) * 256;
      xb[wg * 128 + a_row] = mloc;
      mbar_arrive(bar(B_XCH + wq));
      if (!(ok = warp_wait(bar(B_XCH + wq), n & 1, 18))) break;
      const float mx = fmaxf(mloc, xb[(1 - wg) * 128 + a_row]);
      float corr = 1.f;
      bool rescale_o = false;
      if (mx > m_ref + kRescaleThreshold || (m_ref == -INFINITY && mx != -INFINITY)) {
        const float m_new = fmaxf(m_ref, mx);
        corr = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - m_new);
        rescale_o = (n > 0) && (m_ref != -INFINITY);
        l *= corr;
        m_ref = m_new;
      }
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      {
        uint32_t pk[16];
        float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float e0 = fast_exp2(x[2 * i] - m_use), e1 = fast_exp2(x[2 * i + 1] - m_use);
          rs0 += e0;
          rs1 += e1;
          pk[i] = pack_bf16x2(e0, e1);
        }
        l += rs0 + rs1;
        __syncwarp();
        tmem_st16(sbuf + 16u * wg, pk);   // P (bf16 pairs) over S columns [16 wg, 16 wg + 16)
      }
      // O is only touched when some row of this warp needs a rescale; then PV(n-1)
      // must have landed first.  Otherwise PV(n) simply queues behind PV(n-1)
      // on the tensor core.  (PV completions alternate between two barriers by
      // tile parity; S(n) landing implies PV(n-2) did, so each wait is for the
      // next phase of its barrier and never ambiguous.)
      // TMEM loads / stores are warp-collective: the whole warp rescales its 32
      // rows when any of them needs it (rows that do not are scaled by 1)
      if (__any_sync(0xffffffffu, rescale_o)) {
        if (!(ok = warp_wait(bar(B_PV_DONE + ((n - 1) & 1)), ((n - 1) >> 1) & 1, 16))) break;
        tc_fence_after();
        const float cf = rescale_o ? corr : 1.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          const uint32_t oaddr = tmem + lane_base + TM_O + 64u * wg + 32u * c;
          __syncwarp();
          tmem_ld32(oaddr, r);
          tmem_wait_ld(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * cf);
          __syncwarp();
          tmem_st32(oaddr, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_P_FULL + (n & 1)));
    }
    // ---- epilogue
    if (ok && ntiles > 0)
      ok = warp_wait(bar(B_PV_DONE + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1, 17);
    if (ok) {
      // total row sum over both key halves
      float *xb = xbuf + (ntiles & 1) * 256;
      xb[wg * 128 + a_row] = l;
      mbar_arrive(bar(B_XCH + wq));
      ok = warp_wait(bar(B_XCH + wq), ntiles & 1, 19);
    }
    if (ok) {
      const float lt = l + xbuf[(ntiles & 1) * 256 + (1 - wg) * 128 + a_row];
      tc_fence_after();
      const bool valid = a_row < nrows;
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float row_lse = lt > 0.f ? (m_ref + __log2f(lt)) * kLn2 : -INFINITY;
      const size_t qrow = (size_t)(cq + t_row) * a.Hq + h_row;
      // decode with several splits leaves fp32 partials for the combine kernel
      const bool partial = DECODE && a.num_splits > 1;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        if (ntiles > 0) {
          __syncwarp();
          tmem_ld32(tmem + lane_base + TM_O + 64u * wg + 32u * c, r);
          tmem_wait_ld(r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;   // an empty split contributes nothing
        }
        if (valid && partial) {
          float *dst = a.o_part + ((size_t)split * a.total_q * a.Hq + qrow) * kHeadDim + 64 * wg + 32 * c;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4 *>(dst + 4 * i) =
                make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                            __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
        } else if (valid) {
          __nv_bfloat16 *dst = a.out + qrow * kHeadDim + 64 * wg + 32 * c;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(r[8 * i + 0]) * inv, __uint_as_float(r[8 * i + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(r[8 * i + 2]) * inv, __uint_as_float(r[8 * i + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(r[8 * i + 4]) * inv, __uint_as_float(r[8 * i + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(r[8 * i + 6]) * inv, __uint_as_float(r[8 * i + 7]) * inv);
            *reinterpret_cast<uint4 *>(dst + 8 * i) = v;
          }
        }
      }
      if (valid && wg == 0) {
        if (partial) a.lse_part[(size_t)split * a.total_q * a.Hq + qrow] = row_lse;
        else a.lse[(size_t)h_row * a.total_q + cq + t_row] = row_lse;
      }
    }
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) atomicOr(a.err, kDevErrTimeout | (*abort_flag << 8));
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
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

bool encode(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
            const cuuint64_t *strides, const cuuint32_t *box) {
  auto fn = get_encoder();
  if (!fn) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_supported(const KernelArgs &a, int total_k) {
  auto al = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!get_encoder()) return false;
  if (!al(a.k) || !al(a.v) || !al(a.q) || !al(a.out)) return false;
  if (a.rd > 0) {
    if (a.rd % 8 != 0 || a.E % 8 != 0 || a.rd > 64 || !al(a.r) || !al(a.P)) return false;
  }
  if (total_k < BN) return false;   // K/V boxes stay inside the tensor
  return true;
}

namespace {

template <bool DECODE>
cudaError_t launch_tc(const KernelArgs &a, int total_k, dim3 grid, cudaStream_t stream) {
  TcArgs ta;
  ta.a = a;
  ta.has_bias = a.rd > 0 && a.E > 0;
  CUtensorMap mk, mv;
  {
    cuuint64_t dims[3] = {128, (cuuint64_t)a.Hkv, (cuuint64_t)total_k};
    cuuint64_t strides[2] = {256, (cuuint64_t)a.Hkv * 256};
    cuuint32_t box[3] = {64, 1, BN};
    if (!encode(&mk, a.k, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!encode(&mv, a.v, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(relattn_fwd_tc_kernel<DECODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  relattn_fwd_tc_kernel<DECODE><<<grid, NTHREADS, SMEM_BYTES, stream>>>(ta, mk, mv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const KernelArgs &a, int total_k, cudaStream_t stream) {
  return launch_tc<false>(a, total_k, dim3(a.q_tiles, a.Hq, a.batch), stream);
}

cudaError_t launch_decode_tc(const KernelArgs &a, int total_k, cudaStream_t stream) {
  return launch_tc<true>(a, total_k, dim3(a.num_splits, a.Hkv * a.row_blocks, a.batch), stream);
}

}  // namespace relattn
