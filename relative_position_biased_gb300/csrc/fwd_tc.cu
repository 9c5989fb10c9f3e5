// fwd_tc.cu -- relative-attention forward on 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory, TMA-fed K/V), prefill and
// split-KV decode.
//
// Same computation as the definition on the page "SGLang and Miles Add Day-0
// Support for Inkling", section "Attention with Relative Positional
// Embedding":  x(i,j) = s(i) * (alpha q_i.k_j + [0 <= i-j < E] r_i . P[:, i-j]),
// online softmax, PV.
//
// A work item = 128 query rows (TMEM lane a <-> row a): prefill takes one
// query head x 128 consecutive rows; decode takes 128 rows of the (token,
// head-in-group) list of one kv head and one split of its keys.  Decode and
// the one-launch prefill run one item per CTA; the bias band of the
// two-launch prefill runs one CTA per SM that walks the items, its barrier
// phases and stage rings running on from item to item, so the next item's
// loads and first MMAs overlap the current item's epilogue.  Keys come in
// 128-key tiles (one TMA stage), visited from the diagonal backwards.  Tiles
// inside the relative-bias band are processed as two 64-key half steps (the
// upper half first); the rest as one 128-key step.  Warp roles (12 warps,
// one support and two softmax warps per SM sub-partition; the support warps
// hand registers to the softmax warps in prefill: 88 vs 208 per thread):
//   warp 0      TMA producer (one thread) of K tiles (2-stage ring of 128
//               keys), V tiles (3-stage ring) and P slices P[:, 64c..64c+64)
//               (4 stages), in the order the MMA issuer consumes them; K and
//               V stages are freed separately (K once its S MMAs are done, V
//               after PV).  In the band-only prefill it also loads each
//               item's q rows (into a K-ring slot ahead of the item's tiles)
//               and r rows (into the r tile)
//   warp 1      TMEM allocator; MMA issuer (the warp runs the issue code,
//               an elected lane issues):  S = Q K^T (Q in
//               TMEM; in the band-only prefill copied there from its K-ring
//               slot with tcgen05.cp), R_chunk = r P_slice (both operands from
//               shared memory), O += P V (P in TMEM)
//   warps 2-3   idle
//   warps 4-11  softmax, two warpgroups: row a is owned by one thread of each
//               (TMEM lane a); warpgroup wg takes the lower / upper half of
//               every step's keys.  They write the q / r rows (unless the
//               producer brings them), load S from
//               TMEM, add the relative bias, mask edge tiles, agree on the
//               running row max through shared memory, write P (bf16) back
//               over S, rescale their half of O when the max grows by more
//               than 2^8, and write out / lse (or decode partials) at the end.
//
// Tensor memory (512 columns): Q [0,64) bf16 and O [64,192) always.  During
// the band: half-step S buffers H0 [192,256), H1 [256,320) and the R ring
// [320,512) (three 64-distance chunks of r.P); a half step's P (bf16) is
// written over its S.  After the band: full-step S buffers S0 [192,320),
// S1 [320,448) and one P buffer [448,512), so an S buffer is free as soon as
// the softmax has read it and S(s+2) is computed while step s is in the
// softmax.  The switch happens once per CTA: the first full steps' S are
// issued only after the last half step's P is in.
//
// Relative bias without a sheared tensor: a 64-key half step at offset
// D = i_0 - j_0 needs distances D-63 .. D+span (span = rows' position spread),
// i.e. at most three consecutive 64-distance chunks; walking away from the
// diagonal needs one new chunk per half step.  Each thread loads a window of
// its own row of R (one load shape for the whole warp) and shifts it by its
// lane's offset with a select network, which turns "distance order" into
// "key order" in registers.
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
constexpr int BN = kTcKeyTile;   // keys per tile / TMA stage (128)
constexpr int HN = 64;           // keys per half step (bias band); also the r.P chunk width
constexpr int K_STAGES = 2, V_STAGES = 3;
constexpr int P_STAGES = 4;
constexpr int NTHREADS = 384;
// registers per thread: 168 at launch.  Prefill: the support warpgroup drops
// to 88 and the two softmax warpgroups rise to 208 (4 x 32 x 88 + 8 x 32 x 208
// = 384 x 168).  Decode keeps 168 everywhere (it fits without spills, and
// measured faster).
constexpr uint32_t kRegsSupport = 88, kRegsSoftmax = 208;
static_assert(128 * kRegsSupport + 256 * kRegsSoftmax <= NTHREADS * 168, "register split");
constexpr float kRescaleThreshold = 8.f;   // log2 units

// TMEM columns
constexpr uint32_t TM_Q = 0, TM_O = 64, TM_H = 192, TM_R = 320, TM_S = 192, TM_P = 448;

// Shared memory layout (offsets from a 1024-aligned base).  A K or V stage
// holds two 16 KB boxes [64 dims x 128 keys] (128-byte rows).
constexpr uint32_t KV_BOX_BYTES = 16384;
constexpr uint32_t KV_STAGE_BYTES = 2 * KV_BOX_BYTES;
constexpr uint32_t SM_K = 0;
constexpr uint32_t SM_V = SM_K + K_STAGES * KV_STAGE_BYTES;
constexpr uint32_t SM_RT = SM_V + V_STAGES * KV_STAGE_BYTES;    // r tile 16K
constexpr uint32_t SM_PS = SM_RT + 16384;                      // P slices 4 x 8K
constexpr uint32_t SM_BAR = SM_PS + P_STAGES * 8192;
// barriers (8 bytes each); S_FULL: [0,1] half steps, [2,3] full steps;
// P_FULL: [0,1] half steps; full steps: S_READ, and per warpgroup w P_HALF
// [2w, 2w+1] and PV_F [2w, 2w+1] by step parity.  PV_SW / PV_TAIL are
// committed once each (see the MMA issuer).
constexpr int B_K_FULL = 0, B_K_EMPTY = B_K_FULL + K_STAGES, B_V_FULL = B_K_EMPTY + K_STAGES,
              B_V_EMPTY = B_V_FULL + V_STAGES, B_PS_FULL = B_V_EMPTY + V_STAGES,
              B_PS_EMPTY = B_PS_FULL + P_STAGES, B_RT_FULL = B_PS_EMPTY + P_STAGES,
              B_Q_READY = B_RT_FULL + 1, B_S_FULL = B_Q_READY + 1, B_P_FULL = B_S_FULL + 4,
              B_PV_SW = B_P_FULL + 4, B_PV_TAIL = B_PV_SW + 1, B_R_FULL = B_PV_TAIL + 2,
              B_R_FREE = B_R_FULL + 3, B_S_READ = B_R_FREE + 1, B_PV_F = B_S_READ + 2,
              B_P_HALF = B_PV_F + 4,
              B_DRAIN = B_P_HALF + 4, B_XCH = B_DRAIN + 1, B_RT_EMPTY = B_XCH + 4,
              B_COUNT = B_RT_EMPTY + 1;
constexpr uint32_t SM_TMEM_SLOT = SM_BAR + B_COUNT * 8;
constexpr uint32_t SM_ABORT = SM_TMEM_SLOT + 8;
constexpr uint32_t SM_XCH = SM_ABORT + 8;                      // row exchange [2][2][128] f32
// cu_seqlens_q / _k of up to kCuCache sequences, read once per CTA (the
// persistent CTAs look them up for every item)
constexpr int kCuCache = 64;
constexpr uint32_t SM_CU = SM_XCH + 2 * 2 * 128 * 4;            // [2][kCuCache + 1] int
constexpr uint32_t SM_QLOADS = SM_CU + 2 * (kCuCache + 1) * 4;   // q staging loads issued
// decode work order (batch <= kCuCache): per sequence its full / partial /
// remaining split counts, their prefix sums, and the partial chunks by size
constexpr uint32_t SM_ORD = SM_QLOADS + 8;
constexpr int ORD_NF = 0, ORD_REM = kCuCache, ORD_PF = 2 * kCuCache, ORD_PZ = 3 * kCuCache + 1,
              ORD_PTAB = 4 * kCuCache + 2, ORD_NP = 5 * kCuCache + 2, ORD_INTS = 5 * kCuCache + 4;
constexpr uint32_t SM_TOTAL = SM_ORD + ORD_INTS * 4;
constexpr uint32_t SMEM_BYTES = SM_TOTAL + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct TcArgs {
  KernelArgs a;
  int has_bias;
  // prefill, bias band alone: the q and r rows of an item come by TMA (q
  // into a K-ring slot, copied to TMEM by the MMA issuer; r straight into
  // the r tile), so a CTA's next item starts without the softmax warps
  int stage_tma;
};

__device__ __forceinline__ int floor_div64(int x) { return x >= 0 ? x >> 6 : -((63 - x) >> 6); }

// P of one step's keys for this thread: e = 2^(x c - m) (x raw scores, c > 0),
// packed to bf16 pairs; returns the sum.  All exponentials go to MUFU: the FMA
// pipe is what the MMA-issuing warp competes for on its sub-partition.
template <int NX>
__device__ __forceinline__ float exp_pack_raw(const float (&x)[NX], float c, float m_use,
                                              uint32_t (&pk)[NX / 2]) {
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < NX / 2; ++i) {
    float y0, y1, e0, e1;
    ffma2(y0, y1, x[2 * i], x[2 * i + 1], c, c, -m_use, -m_use);
    e0 = fast_exp2(y0);
    e1 = fast_exp2(y1);
    ffma2(acc[2 * (i & 1)], acc[2 * (i & 1) + 1], e0, e1, 1.f, 1.f, acc[2 * (i & 1)], acc[2 * (i & 1) + 1]);
    pk[i] = pack_bf16x2(e0, e1);
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// max of N values as a tree of three-input maxima (short dependency chains)
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

// One unit of work: 128 query rows and the key tiles they visit.
struct Item {
  int b, kv_head, row0, nrows, split, h_fixed;
  int cq, ck, off, p0, p_last;
  int ntiles, Dt0, span, nb_tiles, s2, nsteps;
  int c_start, c_first, c_last;   // r.P chunks of the band (s2 > 0)
};

template <bool DECODE, bool WALK>
__global__ void __launch_bounds__(NTHREADS, 1)
relattn_fwd_tc_kernel(const __grid_constant__ TcArgs ta,
                      const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v,
                      const __grid_constant__ CUtensorMap map_p,
                      const __grid_constant__ CUtensorMap map_q,
                      const __grid_constant__ CUtensorMap map_r) {
  const KernelArgs &a = ta.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sb = smem_addr(smem);
  auto bar = [&](int i) { return sb + SM_BAR + 8u * i; };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM_ABORT);
  int *cu_s = reinterpret_cast<int *>(smem + SM_CU);   // filled before the set-up barrier
  volatile int *q_loads = reinterpret_cast<volatile int *>(smem + SM_QLOADS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ------------------------------------------------------------ work items
  // Decode: one item per CTA (a split of one kv head's row block).  Prefill:
  // items are (row tile, sequence, head), row tiles from the last (longest
  // running) backwards; CTA x takes items x, x + gridDim.x, ...  Every role
  // walks the same list, and the barrier phases run on across items.
  Item I{};
  // Decode: items are (sequence, split, kv head, row block); CTAs walk them
  // like the prefill's, in longest-first order (see load_item)
  // (WALK = false: decode with one item per CTA, the item from blockIdx)
  const int dec_units = DECODE ? a.Hkv * a.row_blocks : 1;
  const int n_items = DECODE ? (WALK ? a.num_splits * dec_units * a.batch : 1) : a.q_tiles * a.Hq * a.batch;
  const int item0 = (DECODE && !WALK) ? 0 : (int)blockIdx.x;
  const int item_step = (DECODE && !WALK) ? 1 : (int)gridDim.x;
  int *ord = reinterpret_cast<int *>(smem + SM_ORD);
  const bool dec_sorted = DECODE && WALK && a.batch <= kCuCache;
  // work of the items before the current one, for barrier phases / stages
  int hb = 0, fb = 0, tb = 0, ob = 0;     // half steps, full steps, key tiles, r.P chunks
  // V-ring slots: the item's q rows take one ahead of its value tiles (TMA
  // staging; the V ring is the deeper one, so the next item's first K tiles
  // are not held up)
  const int q_slot = (!DECODE && ta.stage_tma) ? 1 : 0;
  int vb = 0;
  auto vslot = [&](int t) { return vb + q_slot + t; };
  int n_it = 0, n_rt = 0;                   // items; items with a band (r tile)
  int n_tail0 = 0, n_tail1 = 0, n_sw = 0;   // PV_TAIL[0/1] and PV_SW commits
  // row (local, clamped to the last valid one) -> token t and query head
  auto row_t = [&](int rl) {
    const int x = I.row0 + min(rl, I.nrows - 1);
    return DECODE ? x / a.group : x;
  };
  auto row_h = [&](int rl) {
    const int x = I.row0 + min(rl, I.nrows - 1);
    return DECODE ? I.kv_head * a.group + x % a.group : I.h_fixed;
  };
  auto tile_D = [&](int t) { return I.Dt0 + BN * t; };
  auto step_tile = [&](int s) { return s < I.s2 ? s >> 1 : I.nb_tiles + (s - I.s2); };
  auto step_kh = [&](int s) { return (s < I.s2 && (s & 1) == 0) ? HN : 0; };   // first key in the tile
  auto step_D = [&](int s) { return tile_D(step_tile(s)) - step_kh(s); };
  // barrier / buffer of a step: half steps alternate 0,1; full steps 2,3 (the
  // half-step count of an item is even, so half steps keep their parity)
  auto step_kind = [&](int s) { return s < I.s2 ? (s & 1) : 2 + ((fb + s - I.s2) & 1); };
  auto step_phase = [&](int s) { return s < I.s2 ? ((hb + s) >> 1) & 1 : ((fb + s - I.s2) >> 1) & 1; };
  // full-step index across items (S_READ / P_HALF / PV_F parity and phase)
  auto full_idx = [&](int s) { return fb + s - I.s2; };
  // newest r.P chunk (64 distances) a half step needs: one more per half step
  auto c_new = [&](int s) { return floor_div64(step_D(s) + I.span); };
  // chunk c of the current item: ring slot / P stage / barrier phase index
  auto chunk_idx = [&](int c) { return ob + (c - I.c_start); };
  // 1 = work to do, 0 = nothing (row tile past the sequence, empty split),
  // -1 = inconsistent sequence lengths (reported by the caller, item skipped)
  auto load_item = [&](int idx) -> int {
    if constexpr (DECODE) {
      // slot idx -> position: rounds of gridDim.x slots, every other full round
      // reversed (a snake), over pairs (sequence, split) ordered full chunks
      // first, then partial chunks by size, then the rest; each pair is
      // dec_units consecutive items (kv head, row block).  Every pair is in
      // the order, so the walk covers all items whatever the sizes.
      int b, sp, u;
      if constexpr (!WALK) {
        sp = blockIdx.x;
        u = blockIdx.y;
        b = blockIdx.z;
      } else if (dec_sorted) {
        const int r = idx / item_step, c = idx - r * item_step;
        const int pos = ((r & 1) && (r + 1) * item_step <= n_items) ? r * item_step + (item_step - 1 - c) : idx;
        const int q = pos / dec_units;
        u = pos - q * dec_units;
        const int F = ord[ORD_PF + a.batch], NP = ord[ORD_NP];
        if (q < F || q >= F + NP) {
          const int base = q < F ? ORD_PF : ORD_PZ, qq = q < F ? q : q - F - NP;
          b = 0;                                        // last b with prefix[b] <= qq
          for (int i = 1; i < a.batch; ++i) b = ord[base + i] <= qq ? i : b;
          sp = q < F ? qq - ord[ORD_PF + b]
                     : ord[ORD_NF + b] + (ord[ORD_REM + b] > 0 ? 1 : 0) + (qq - ord[ORD_PZ + b]);
        } else {
          b = ord[ORD_PTAB + (q - F)];
          sp = ord[ORD_NF + b];
        }
      } else {
        sp = idx % a.num_splits;
        const int rest = idx / a.num_splits;
        u = rest % dec_units;
        b = rest / dec_units;
      }
      I.split = sp;
      I.kv_head = u / a.row_blocks;
      I.row0 = (u % a.row_blocks) * BM;
      I.b = b;
      I.h_fixed = 0;
    } else {
      const int per_x = a.Hq * a.batch;
      const int xi = idx / per_x, rem = idx - xi * per_x;
      I.b = rem / a.Hq;
      I.h_fixed = rem - I.b * a.Hq;
      I.split = 0;
      I.kv_head = I.h_fixed / a.group;
      I.row0 = (a.q_tiles - 1 - xi) * BM;
    }
    const int *cuq = a.batch <= kCuCache ? cu_s : a.cu_q;
    const int *cuk = a.batch <= kCuCache ? cu_s + kCuCache + 1 : a.cu_k;
    I.cq = cuq[I.b];
    I.ck = cuk[I.b];
    const int Lq = cuq[I.b + 1] - I.cq, Lk = cuk[I.b + 1] - I.ck;
    if (Lq < 0 || Lk < Lq || Lq > a.max_q || Lk > a.max_k) return -1;
    I.nrows = min(BM, (DECODE ? Lq * a.group : Lq) - I.row0);
    if (I.nrows <= 0) return 0;
    I.off = Lk - Lq;
    I.p0 = I.off + row_t(0);
    I.p_last = I.off + row_t(I.nrows - 1);
    const int j_lo = a.window > 0 ? max(0, I.p0 - a.window + 1) : 0;
    // 128-key tiles from the diagonal backwards: tile t starts at key
    // p0 - D(t); the rows sit at positions p0 + delta, 0 <= delta <= span
    if constexpr (DECODE) {
      const int kbase = j_lo & ~(BN - 1);
      const int kbeg = kbase + I.split * a.split_chunk;
      const int kend = min(I.p_last + 1, kbeg + a.split_chunk);
      I.ntiles = kend > kbeg ? (kend - kbeg + BN - 1) / BN : 0;
      I.Dt0 = I.p0 - (kbeg + (I.ntiles - 1) * BN);
      I.span = I.p_last - I.p0;
    } else {
      I.Dt0 = 0;                                   // tile 0 = keys [p0, p0 + 127]
      I.ntiles = (I.p0 - j_lo + BN - 1) / BN + 1;
      I.span = BM - 1;   // padding rows reuse the pattern of full tiles
    }
    // band tiles (some distance < E) form a prefix of the tile order
    I.nb_tiles = 0;
    if (ta.has_bias && I.ntiles > 0) {
      const int lim = a.E + BN - 1;              // band iff D - 127 < E
      I.nb_tiles = tile_D(I.ntiles - 1) < lim ? I.ntiles : max(0, (lim - I.Dt0 + BN - 1) / BN);
      if (I.nb_tiles > I.ntiles) I.nb_tiles = I.ntiles;
    }
    // prefill split in two kernels: this one takes only the band, and leaves
    // out / lse normalised over the band's keys for the main kernel to continue
    if (!DECODE && a.band_only && I.nb_tiles > 0) I.ntiles = I.nb_tiles;
    I.s2 = 2 * I.nb_tiles;                         // first full step
    I.nsteps = I.s2 + (I.ntiles - I.nb_tiles);
    I.c_first = I.s2 > 0 ? c_new(0) : -1;
    I.c_last = I.s2 > 0 ? c_new(I.s2 - 1) : -1;
    // first chunk computed: the oldest one step 0 reads (a decode split far
    // from the diagonal starts deep in the band)
    I.c_start = I.s2 > 0 ? max(0, floor_div64(step_D(0) - (HN - 1))) : 0;
    return 1;
  };
  // after an item: advance the cross-item counters (every role, same values)
  auto finish_item = [&]() {
    hb += I.s2;
    fb += I.nsteps - I.s2;
    tb += I.ntiles;
    vb += I.ntiles + q_slot;
    ob += I.s2 > 0 ? I.c_last - I.c_start + 1 : 0;
    n_tail0 += I.nsteps >= 2;
    n_tail1 += I.nsteps >= 1;
    n_sw += (I.s2 > 0 && I.s2 < I.nsteps);
    n_rt += I.s2 > 0;
    ++n_it;
  };

  // ------------------------------------------------------------ setup
  if (tid == 0) {
    for (int i = 0; i < K_STAGES; ++i) {
      mbar_init(bar(B_K_FULL + i), 1);
      mbar_init(bar(B_K_EMPTY + i), 1);
    }
    for (int i = 0; i < V_STAGES; ++i) {
      mbar_init(bar(B_V_FULL + i), 1);
      mbar_init(bar(B_V_EMPTY + i), 1);
    }
    for (int i = 0; i < P_STAGES; ++i) {
      mbar_init(bar(B_PS_FULL + i), 1);
      mbar_init(bar(B_PS_EMPTY + i), 1);
    }
    mbar_init(bar(B_RT_FULL), q_slot ? 1 : 256);
    mbar_init(bar(B_RT_EMPTY), 1);
    mbar_init(bar(B_Q_READY), 256);
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(B_S_FULL + i), 1);
      mbar_init(bar(B_P_FULL + i), 256);
    }
    mbar_init(bar(B_PV_SW), 1);
    mbar_init(bar(B_PV_TAIL), 1);
    mbar_init(bar(B_PV_TAIL + 1), 1);
    for (int i = 0; i < 2; ++i) mbar_init(bar(B_S_READ + i), 256);
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(B_PV_F + i), 1);
      mbar_init(bar(B_P_HALF + i), 128);
    }
    for (int i = 0; i < 3; ++i) mbar_init(bar(B_R_FULL + i), 1);
    mbar_init(bar(B_R_FREE), 256);
    mbar_init(bar(B_DRAIN), 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar(B_XCH + i), 64);
    *abort_flag = 0;
    *q_loads = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + SM_TMEM_SLOT, 512);
    tmem_relinquish();
  }
  if (a.batch <= kCuCache && tid >= 128 && tid < 128 + 2 * (a.batch + 1)) {
    const int i = tid - 128;
    cu_s[i <= a.batch ? i : kCuCache + 1 + (i - a.batch - 1)] =
        i <= a.batch ? a.cu_q[i] : a.cu_k[i - a.batch - 1];
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map_k);
    prefetch_tmap(&map_v);
    if (ta.has_bias) prefetch_tmap(&map_p);
    if (q_slot) {
      prefetch_tmap(&map_q);
      prefetch_tmap(&map_r);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (dec_sorted) {
    // the decode work order: sequence b's keys from the aligned start of its
    // first row block's window, cut into splits of split_chunk keys
    const int b = tid;
    if (b < a.batch) {
      const int cq = cu_s[b], ck = cu_s[kCuCache + 1 + b];
      const int Lq = cu_s[b + 1] - cq, Lk = cu_s[kCuCache + 2 + b] - ck;
      long vis = 0;
      if (Lq > 0 && Lk >= Lq) {
        const int off = Lk - Lq, rows = min(BM, Lq * a.group);
        const int p0 = off, p_last = off + (rows - 1) / a.group;
        const int j_lo = a.window > 0 ? max(0, p0 - a.window + 1) : 0;
        vis = (long)p_last + 1 - (j_lo & ~(BN - 1));
      }
      const long nf = min((long)a.num_splits, vis / a.split_chunk);
      const long rem = nf < a.num_splits ? vis - nf * a.split_chunk : 0;
      ord[ORD_NF + b] = (int)nf;
      ord[ORD_REM + b] = (int)rem;
    }
    __syncthreads();
    if (tid == 0) {
      int f = 0, z = 0, np = 0;
      for (int i = 0; i < a.batch; ++i) {
        ord[ORD_PF + i] = f;
        ord[ORD_PZ + i] = z;
        const int pi = ord[ORD_REM + i] > 0 ? 1 : 0;
        f += ord[ORD_NF + i];
        z += a.num_splits - ord[ORD_NF + i] - pi;
        np += pi;
      }
      ord[ORD_PF + a.batch] = f;
      ord[ORD_PZ + a.batch] = z;
      ord[ORD_NP] = np;
    }
    if (b < a.batch && ord[ORD_REM + b] > 0) {   // rank among the partial chunks: larger first
      const int rb = ord[ORD_REM + b];
      int rank = 0;
      for (int i = 0; i < a.batch; ++i) {
        const int ri = ord[ORD_REM + i];
        rank += ri > rb || (ri == rb && i < b);
      }
      ord[ORD_PTAB + rank] = b;
    }
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + SM_TMEM_SLOT);
  // TMA copies issued by the producer thread (to drain them if the CTA gives up)
  int issued_k = 0, issued_v = 0, issued_p = 0, issued_rt = 0;
  if (warp < 4) {
  if constexpr (!DECODE || WALK) regs_dec<kRegsSupport>();
  if (warp == 0) {
    // ======================================================== TMA producer
    // Per tile t: the P slices its half steps need (band tiles), then K(t),
    // then V(t) -- the order the MMA issuer consumes them, so a wait here only
    // ever depends on work issued before it.  A P slice is P[0:r_dim, 64c ..
    // 64c + 64) in the 128-byte-swizzled layout (columns past E read as 0;
    // rows r_dim .. rd_pad stay at the zeros the softmax warps put there).
    // The stage rings run on across items, so the next item's tiles load
    // while the current one finishes.
    if (lane == 0) {
      const uint32_t p_bytes = 128u * (uint32_t)a.rd;
      int kst = 0, kph = 0, vst = 0, vph = 0;
      bool run = true;
      for (int idx = item0; idx < n_items && run; idx += item_step) {
        const int li = load_item(idx);
        if (li < 0) atomicOr(a.err, kDevErrSeqlens);
        if (li <= 0) continue;
        if (q_slot) {
          // q rows -> the item's first V-ring slot (rows past the sequence
          // read other rows or zeros: padding rows, never stored); first,
          // since the r tile waits for the previous item's last r.P chunk
          if (vb >= V_STAGES && !(run = mbar_wait(bar(B_V_EMPTY + vst), vph ^ 1, abort_flag, 4))) break;
          const uint32_t dst = sb + SM_V + vst * KV_STAGE_BYTES;
          mbar_arrive_expect_tx(bar(B_V_FULL + vst), KV_STAGE_BYTES);
          tma_load_3d(dst, &map_q, 0, I.h_fixed, I.cq + I.row0, bar(B_V_FULL + vst));
          tma_load_3d(dst + KV_BOX_BYTES, &map_q, 64, I.h_fixed, I.cq + I.row0, bar(B_V_FULL + vst));
          issued_v = vb + 1;
          *q_loads = n_it + 1;   // q rows of this CTA's first n_it + 1 items are on their way
          if (++vst == V_STAGES) { vst = 0; vph ^= 1; }
          // r rows -> r tile, once the previous item's r.P chunks are done
          if (I.s2 > 0) {
            if (n_rt > 0 && !(run = mbar_wait(bar(B_RT_EMPTY), (n_rt - 1) & 1, abort_flag, 20))) break;
            mbar_arrive_expect_tx(bar(B_RT_FULL), 16384u);
            tma_load_3d(sb + SM_RT, &map_r, 0, I.h_fixed, I.cq + I.row0, bar(B_RT_FULL));
            issued_rt = n_rt + 1;
          }
        }
        int c_next = I.c_start;
        // paged decode: pool page of tile t's keys
        auto page_of = [&](int t) {
          return a.block_table[(size_t)I.b * a.max_pages + (I.p0 - tile_D(t)) / a.page_size];
        };
        int pg_next = (DECODE && a.block_table != nullptr && I.ntiles > 0) ? page_of(0) : 0;
        for (int t = 0; t < I.ntiles && run && !*abort_flag; ++t) {
          if (t < I.nb_tiles) {
            const int c_need = c_new(2 * t + 1);   // newest chunk of the tile's second half step
            for (; c_next <= c_need; ++c_next) {
              const int o = chunk_idx(c_next), st = o % P_STAGES;
              if (o >= P_STAGES &&
                  !(run = mbar_wait(bar(B_PS_EMPTY + st), ((o / P_STAGES) - 1) & 1, abort_flag, 3)))
                break;
              mbar_arrive_expect_tx(bar(B_PS_FULL + st), p_bytes);
              tma_load_2d(sb + SM_PS + st * 8192, &map_p, HN * c_next, 0, bar(B_PS_FULL + st));
              issued_p = o + 1;
            }
            if (!run) break;
          }
          const int kg = tb + t, vg = vslot(t);        // K / V ring index across items
          int key = I.ck + I.p0 - tile_D(t);           // may be < 0: the tile reads zeros there
          if constexpr (DECODE) {
            if (a.block_table != nullptr) {
              // paged: the tile (128-aligned, inside one page) -> its pool rows;
              // a page number outside the pool reads zeros and is reported.
              // The next tile's entry is read now, to land during this tile's waits.
              const int p = I.p0 - tile_D(t);
              const int pg = pg_next;
              if (t + 1 < I.ntiles) pg_next = page_of(t + 1);
              const bool ok = pg >= 0 && pg < a.num_pages;
              if (!ok) atomicOr(a.err, kDevErrSeqlens);
              key = ok ? pg * a.page_size + p % a.page_size : -BN;
            }
          }
          if (kg >= K_STAGES && !(run = mbar_wait(bar(B_K_EMPTY + kst), kph ^ 1, abort_flag, 1))) break;
          if (kg != a.test_skip_k_tile) {   // (test hook: a skipped tile is never loaded)
            const uint32_t dst = sb + SM_K + kst * KV_STAGE_BYTES;
            mbar_arrive_expect_tx(bar(B_K_FULL + kst), KV_STAGE_BYTES);
            tma_load_3d(dst, &map_k, 0, I.kv_head, key, bar(B_K_FULL + kst));
            tma_load_3d(dst + KV_BOX_BYTES, &map_k, 64, I.kv_head, key, bar(B_K_FULL + kst));
          }
          issued_k = kg + 1;
          if (++kst == K_STAGES) { kst = 0; kph ^= 1; }
          if (vg >= V_STAGES && !(run = mbar_wait(bar(B_V_EMPTY + vst), vph ^ 1, abort_flag, 4))) break;
          {
            const uint32_t dst = sb + SM_V + vst * KV_STAGE_BYTES;
            mbar_arrive_expect_tx(bar(B_V_FULL + vst), KV_STAGE_BYTES);
            tma_load_3d(dst, &map_v, 0, I.kv_head, key, bar(B_V_FULL + vst));
            tma_load_3d(dst + KV_BOX_BYTES, &map_v, 64, I.kv_head, key, bar(B_V_FULL + vst));
            issued_v = vg + 1;
            if (++vst == V_STAGES) { vst = 0; vph ^= 1; }
          }
        }
        if (*abort_flag) run = false;
        finish_item();
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================================================== MMA issuer
    // The whole warp runs the issue code (descriptors stay warp-uniform); each
    // MMA, copy and commit is issued by one elected lane.
    {
      const uint32_t id_h = idesc_bf16_f32(BM, HN, 0, 0);       // half S: Q(tmem) x K(smem, K-major)
      const uint32_t id_f = idesc_bf16_f32(BM, BN, 0, 0);       // full S
      const uint32_t id_o = idesc_bf16_f32(BM, 128, 0, 1);      // O: P(tmem) x V(smem, MN-major)
      const uint32_t id_r = idesc_bf16_f32(BM, HN, 0, 1);       // R: r(smem) x P(smem, MN-major)
      const int r_ksteps = a.rd_pad / 16;
      // descriptor bases; per k-step / stage / half only the 16-byte address
      // field moves: +2 per 32 bytes of a 128-byte row, +1024 per 16 KB box,
      // +8 per key row, +128 per 16 V rows
      const uint64_t kd0 = smem_desc_sw128(sb + SM_K, 16, 1024);
      const uint64_t vd0 = smem_desc_sw128(sb + SM_V, KV_BOX_BYTES, 1024);
      const uint64_t rd0 = smem_desc_sw128(sb + SM_RT, 16, 1024);
      const uint64_t pd0 = smem_desc_sw128(sb + SM_PS, 8192, 1024);
      bool ok = true;
      bool rt_ready = false;
      // q rows of an item: V-ring slot vq -> TMEM (eight 128x256b copies, in
      // the same 128-byte-swizzled K-major layout as a K tile), then the slot
      // is free again.  Every S MMA that read the previous q has landed.
      auto copy_q = [&](int vq) -> bool {
        const int st = vq % V_STAGES;
        if (!mbar_wait_warp(bar(B_V_FULL + st), (vq / V_STAGES) & 1, abort_flag, 6)) return false;
        tc_fence_after();
        const uint64_t qd = kd0 + (uint64_t)((SM_V - SM_K + st * KV_STAGE_BYTES) >> 4);
        tmem_cp_128x256b_e(tmem + TM_Q + 0, qd + 0);
        tmem_cp_128x256b_e(tmem + TM_Q + 8, qd + 2);
        tmem_cp_128x256b_e(tmem + TM_Q + 16, qd + 4);
        tmem_cp_128x256b_e(tmem + TM_Q + 24, qd + 6);
        tmem_cp_128x256b_e(tmem + TM_Q + 32, qd + 1024);
        tmem_cp_128x256b_e(tmem + TM_Q + 40, qd + 1026);
        tmem_cp_128x256b_e(tmem + TM_Q + 48, qd + 1028);
        tmem_cp_128x256b_e(tmem + TM_Q + 56, qd + 1030);
        mma_commit_e(bar(B_V_EMPTY + st));
        return true;
      };
      bool q_in = false;   // the current item's q rows are already in TMEM
      auto issue_r = [&](int c) -> bool {
        if (!rt_ready) {
          if (!mbar_wait_warp(bar(B_RT_FULL), n_rt & 1, abort_flag, 7)) return false;
          rt_ready = true;
        }
        const int o = chunk_idx(c);
        const int st = o % P_STAGES;
        if (!mbar_wait_warp(bar(B_PS_FULL + st), (o / P_STAGES) & 1, abort_flag, 8)) return false;
        tc_fence_after();
        const uint32_t d = tmem + TM_R + 64u * (uint32_t)(o % 3);
        const uint64_t pd = pd0 + (uint64_t)((st * 8192) >> 4);
        mma_ss_e<0>(d, rd0, pd, id_r);
        if (r_ksteps > 1) mma_ss_e<1>(d, rd0 + 2, pd + 128, id_r);
        if (r_ksteps > 2) mma_ss_e<1>(d, rd0 + 4, pd + 256, id_r);
        if (r_ksteps > 3) mma_ss_e<1>(d, rd0 + 6, pd + 384, id_r);
        mma_commit_e(bar(B_R_FULL + o % 3));
        // the item's last chunk: once it lands the r tile may take the next item's rows
        if (q_slot && c == I.c_last) mma_commit_e(bar(B_RT_EMPTY));   // its landing also frees P stage st (softmax arrives)
        return true;
      };
      auto issue_s = [&](int s) -> bool {
        const int t = tb + step_tile(s), st = t % K_STAGES;
        // (the second half step of a tile uses the K tile the first one waited for)
        if (!(s < I.s2 && (s & 1)) && !mbar_wait_warp(bar(B_K_FULL + st), (t / K_STAGES) & 1, abort_flag, 9))
          return false;
        tc_fence_after();
        const uint32_t qa = tmem + TM_Q;
        const uint64_t kd = kd0 + (uint64_t)((st * KV_STAGE_BYTES) >> 4) + (uint64_t)(step_kh(s) * 8);
        // k-step k: dims 16k..16k+15 -> box k/4, 32 bytes per step inside the row
        if (s < I.s2) {
          const uint32_t d = tmem + TM_H + 64u * (uint32_t)(s & 1);
          mma_ts_e<0>(d, qa + 0, kd + 0, id_h);
          mma_ts_e<1>(d, qa + 8, kd + 2, id_h);
          mma_ts_e<1>(d, qa + 16, kd + 4, id_h);
          mma_ts_e<1>(d, qa + 24, kd + 6, id_h);
          mma_ts_e<1>(d, qa + 32, kd + 1024, id_h);
          mma_ts_e<1>(d, qa + 40, kd + 1026, id_h);
          mma_ts_e<1>(d, qa + 48, kd + 1028, id_h);
          mma_ts_e<1>(d, qa + 56, kd + 1030, id_h);
        } else {
          const uint32_t d = tmem + TM_S + 128u * (uint32_t)(full_idx(s) & 1);
          mma_ts_e<0>(d, qa + 0, kd + 0, id_f);
          mma_ts_e<1>(d, qa + 8, kd + 2, id_f);
          mma_ts_e<1>(d, qa + 16, kd + 4, id_f);
          mma_ts_e<1>(d, qa + 24, kd + 6, id_f);
          mma_ts_e<1>(d, qa + 32, kd + 1024, id_f);
          mma_ts_e<1>(d, qa + 40, kd + 1026, id_f);
          mma_ts_e<1>(d, qa + 48, kd + 1028, id_f);
          mma_ts_e<1>(d, qa + 56, kd + 1030, id_f);
        }
        // one commit per S group: its landing also tells the softmax warps that
        // the K stage was read (for the tile's last S) and that every MMA
        // issued before it, PV(s - 2) included, has finished
        mma_commit_e(bar(B_S_FULL + step_kind(s)));
        return true;
      };
      // O += P V; k-step k = 16 keys = 2048 bytes of the MN-major V tile
      auto issue_pv = [&](int s) -> bool {
        const int t = vslot(step_tile(s)), st = t % V_STAGES;
        if (!(s < I.s2 && (s & 1)) && !mbar_wait_warp(bar(B_V_FULL + st), (t / V_STAGES) & 1, abort_flag, 5))
          return false;
        tc_fence_after();
        const uint64_t vd = vd0 + (uint64_t)((st * KV_STAGE_BYTES) >> 4) + (uint64_t)(step_kh(s) * 8);
        const uint32_t o = tmem + TM_O;
        if (s < I.s2) {
          const uint32_t pa = tmem + TM_H + 64u * (uint32_t)(s & 1);
          if (s > 0) mma_ts_e<1>(o, pa + 0, vd + 0, id_o);
          else mma_ts_e<0>(o, pa + 0, vd + 0, id_o);
          mma_ts_e<1>(o, pa + 8, vd + 128, id_o);
          mma_ts_e<1>(o, pa + 16, vd + 256, id_o);
          mma_ts_e<1>(o, pa + 24, vd + 384, id_o);
        } else {
          // two halves, one per warpgroup's P (keys 0..63 / 64..127), each
          // issued as soon as that warpgroup's P is in
          const int par = full_idx(s) & 1, ph = (full_idx(s) >> 1) & 1;
          for (int h = 0; h < 2; ++h) {
            if (!mbar_wait_warp(bar(B_P_HALF + 2 * h + par), ph, abort_flag, 11)) return false;
            tc_fence_after();
            const uint32_t pa = tmem + TM_P + 32u * h;
            const uint64_t vh = vd + 512 * h;
            if (s > 0 || h > 0) mma_ts_e<1>(o, pa + 0, vh + 0, id_o);
            else mma_ts_e<0>(o, pa + 0, vh + 0, id_o);
            mma_ts_e<1>(o, pa + 8, vh + 128, id_o);
            mma_ts_e<1>(o, pa + 16, vh + 256, id_o);
            mma_ts_e<1>(o, pa + 24, vh + 384, id_o);
            // this half of the P buffer is free again once this lands
            mma_commit_e(bar(B_PV_F + 2 * h + par));
          }
        }
        // In the band, PV(s) completion is learnt from the landing of S(s + 2)
        // (or S(s + 1) for an O rescale at step s + 1); commits only where no
        // such S follows without waiting for P: the last two steps, and the step
        // before the first full step (whose S is issued after the last half
        // step's PV).  Full steps commit PV_F above.
        if (s == I.nsteps - 2) mma_commit_e(bar(B_PV_TAIL));
        if (s == I.nsteps - 1) mma_commit_e(bar(B_PV_TAIL + 1));
        if (I.s2 < I.nsteps && s == I.s2 - 2) mma_commit_e(bar(B_PV_SW));
        return true;
      };
      for (int idx = item0; idx < n_items && ok; idx += item_step) {
      if (load_item(idx) <= 0) continue;
      // the item's q (TMEM) and r (shared) rows are in: everything of the
      // previous item that read them has finished (its S / R landings were
      // awaited by the softmax warps first)
      if (q_slot) {
        // the item's q rows, unless they went in during the previous item's
        // last step
        if (q_in) q_in = false;
        else ok = copy_q(vb);
      } else {
        ok = mbar_wait_warp(bar(B_Q_READY), n_it & 1, abort_flag, 6);
        tc_fence_after();
      }
      rt_ready = false;
      if (ok && I.s2 > 0)
        for (int c = I.c_start; c <= I.c_first && ok; ++c) ok = issue_r(c);
      if (ok && I.nsteps > 0) ok = issue_s(0);   // an empty decode split issues nothing
      if (ok && I.s2 == 0 && I.nsteps > 1) ok = issue_s(1);   // full steps keep two S in flight
      // with TMA-staged q rows (band only: every step a half step) the last
      // step comes after the loop
      const int s_loop = q_slot ? I.nsteps - 1 : I.nsteps;
      for (int s = 0; s < s_loop && ok; ++s) {
        if (s < I.s2) {
          // ---- half step: S(s+1) ahead of PV(s).  The first full steps' S
          // buffers overlap the half-step buffers and the R ring: they are
          // issued only once the last half step's P is in.
          const bool switch_next = (s + 1 == I.s2) && (I.s2 < I.nsteps);
          if (!switch_next && s + 1 < I.nsteps && !(ok = issue_s(s + 1))) break;
          if (s + 1 < I.s2) {
            const int c = c_new(s + 1);
            if (!(ok = mbar_wait_warp(bar(B_R_FREE), (hb + s) & 1, abort_flag, 10))) break;
            if (c >= I.c_start && !(ok = issue_r(c))) break;
          }
          if (!(ok = mbar_wait_warp(bar(B_P_FULL + step_kind(s)), step_phase(s), abort_flag, 11))) break;
          tc_fence_after();
          if (!(ok = issue_pv(s))) break;
          if (switch_next) {
            if (!(ok = issue_s(s + 1))) break;
            if (s + 2 < I.nsteps && !(ok = issue_s(s + 2))) break;
          }
        } else {
          // ---- full step: S(s+2) into the buffer of S(s) as soon as the
          // softmax has read it, then PV(s)
          if (s + 2 < I.nsteps) {
            if (!(ok = mbar_wait_warp(bar(B_S_READ + (full_idx(s) & 1)), (full_idx(s) >> 1) & 1, abort_flag, 19))) break;
            tc_fence_after();
            if (!(ok = issue_s(s + 2))) break;
          }
          if (!(ok = issue_pv(s))) break;   // waits for each warpgroup's P half
        }
      }
      if (q_slot && ok && I.nsteps > 0) {
        const int s = I.nsteps - 1;
        // once the last S has landed nothing reads q: the next item's q rows
        // go in now, ahead of this step's PV (if the producer has issued them
        // already; else at the next item's start)
        if (__shfl_sync(0xffffffffu, *q_loads, 0) > n_it + 1) {
          ok = mbar_wait_warp(bar(B_S_FULL + step_kind(s)), step_phase(s), abort_flag, 13);
          tc_fence_after();
          if (ok) ok = copy_q(vb + I.ntiles + q_slot);
          q_in = ok;
        }
        if (ok) ok = mbar_wait_warp(bar(B_P_FULL + step_kind(s)), step_phase(s), abort_flag, 11);
        tc_fence_after();
        if (ok) ok = issue_pv(s);
      }
      finish_item();
      }
      // drain: every MMA issued above has finished before TMEM is released
      mma_commit_e(bar(B_DRAIN));
      volatile int keep_waiting = 0;
      mbar_wait(bar(B_DRAIN), 0, &keep_waiting, 12, 400000000ll);
    }
    __syncwarp();
  }
  } else {
    if constexpr (!DECODE || WALK) regs_inc<kRegsSoftmax>();
    // ======================================================== softmax
    // Two warpgroups share the 128 rows: warpgroup wg handles the wg-th half of
    // every step's keys and O / output columns [64 wg, 64 wg + 64).  The two
    // threads of a row agree on the running max through a shared-memory
    // exchange guarded by a per-lane-quarter mbarrier.
    const int wg = (warp - 4) >> 2;
    const int wq = warp & 3;                     // lane quarter (TMEM lanes 32 wq ..)
    const bool leader = warp == 4 && lane == 0;  // releases K / V / P stages
    const int a_row = 32 * wq + lane;            // row == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    // scores are scaled by cqk > 0: a negative alpha flips the sign of q
    // instead (exact in bf16), so a row max of raw scores is a max of logits
    const bool q_neg = a.alpha_log2e < 0.f;
    float *xbuf = reinterpret_cast<float *>(smem + SM_XCH);   // [2 parity][2 wg][128]
    // every lane of a softmax warp takes the same branch after a wait, so the
    // warp-collective tcgen05 loads / stores that follow see a converged warp
    auto warp_wait = [&](uint32_t br, uint32_t parity, int site) -> bool {
      const bool r = mbar_wait(br, parity, abort_flag, site);
      return __all_sync(0xffffffffu, r);
    };
    // combine this thread's value with the other warpgroup's for the same row
    // (buffer and barrier phase by the parity of the exchange count)
    int n_xch = 0;
    auto exchange = [&](float v, bool &okx) -> float {
      float *xb = xbuf + (n_xch & 1) * 256;
      xb[wg * 128 + a_row] = v;
      mbar_arrive(bar(B_XCH + wq));
      okx = warp_wait(bar(B_XCH + wq), n_xch & 1, 18);
      ++n_xch;
      return xb[(1 - wg) * 128 + a_row];
    };
    bool ok = true;
    int idx = item0;
    // the next item with work (every role walks the same list)
    auto next_item = [&]() -> bool {
      for (; idx < n_items; idx += item_step)
        if (load_item(idx) > 0) {
          idx += item_step;
          return true;
        }
      return false;
    };
    // the current item's q and r rows; once they are in, the MMA issuer may
    // start the item
    auto stage_item = [&]() {
      const int t_row = row_t(a_row), h_row = row_h(a_row);
      // q row half -> TMEM columns [32 wg, 32 wg + 32) (bf16 pairs)
      {
        const uint4 *src = reinterpret_cast<const uint4 *>(
            a.q + ((size_t)(I.cq + t_row) * a.Hq + h_row) * kHeadDim + 64 * wg);
        uint32_t r[32];
  #pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = src[i];
          r[4 * i] = v.x; r[4 * i + 1] = v.y; r[4 * i + 2] = v.z; r[4 * i + 3] = v.w;
        }
        if (q_neg) {
  #pragma unroll
          for (int i = 0; i < 32; ++i) r[i] ^= 0x80008000u;
        }
        __syncwarp();
        tmem_st32(tmem + lane_base + TM_Q + 32u * wg, r);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(B_Q_READY));
      }
      // r row half -> shared r tile (row a, 128-byte swizzle; zero past r_dim)
      if (I.s2 > 0) {
        const __nv_bfloat16 *rsrc = a.r + ((size_t)(I.cq + t_row) * a.Hq + h_row) * a.rd;
        uint8_t *rrow = smem + SM_RT + (a_row >> 3) * 1024 + (a_row & 7) * 128;
  #pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 4 * wg + jj;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (8 * j < a.rd) v = *reinterpret_cast<const uint4 *>(rsrc + 8 * j);
          *reinterpret_cast<uint4 *>(rrow + ((j ^ (a_row & 7)) << 4)) = v;
        }
        // P-slice rows r_dim .. rd_pad of every stage are zero (the TMA box
        // covers r_dim rows); written once, before the first R MMA
        const int zero_chunks = n_rt == 0 ? (a.rd_pad - a.rd) * 8 * P_STAGES : 0;
        for (int i = a_row + 128 * wg; i < zero_chunks; i += 256) {
          const int st = i / ((a.rd_pad - a.rd) * 8), rem = i % ((a.rd_pad - a.rd) * 8);
          const int ch = a.rd + (rem >> 3), j = rem & 7;
          *reinterpret_cast<uint4 *>(smem + SM_PS + st * 8192 + (ch >> 3) * 1024 + (ch & 7) * 128 + j * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(B_RT_FULL));
      }
    };
    bool have = next_item();
    if (have && !q_slot) stage_item();
    while (have && ok) {
    const int t_row = row_t(a_row), h_row = row_h(a_row);
    // position of this row; prefill padding rows (a_row >= nrows) continue the
    // diagonal pattern and only compute garbage that is never stored
    const int pos = DECODE ? I.off + t_row : I.p0 + a_row;
    const int delta = pos - I.p0;                // 0 .. span
    const int delta_w = DECODE ? I.off + row_t(32 * wq) - I.p0 : 32 * wq;   // first row of the warp
    const float sc = log_scale(min(pos, I.p_last), a.inv_ln_base);
    const float cqk = fmaxf(fabsf(a.alpha_log2e) * sc, 1e-30f), cbias = kLog2e * sc;
    // band steps form t = |alpha| S + bias and apply cbias inside the exponent
    const float qk_over_bias = cqk / cbias;

    // TMEM address of distances d0 .. d0+31; valid for chunks >= c_start
    auto r_addr = [&](int d0) {
      return tmem + lane_base + TM_R + 64u * (uint32_t)(chunk_idx(d0 >> 6) % 3) + (uint32_t)(d0 & 63);
    };
    const int d_min = HN * I.c_start;   // smaller distances were never computed (not needed)
    float m_ref = -INFINITY, l = 0.f;
    for (int s = 0; s < I.nsteps; ++s) {
      if (!(ok = warp_wait(bar(B_S_FULL + step_kind(s)), step_phase(s), 13))) break;
      if (leader) {
        // S(s) landed: the K stage of its tile is read (last S of the tile)
        if (step_kh(s) == 0) mbar_arrive(bar(B_K_EMPTY + (tb + step_tile(s)) % K_STAGES));
        // (S(s) is issued after PV(s-2) while s - 2 is a half step; full steps
        // release their V stage after waiting for PV_F instead)
        if (s >= 2 && s - 2 < I.s2 && step_kh(s - 2) == 0)
          mbar_arrive(bar(B_V_EMPTY + vslot(step_tile(s - 2)) % V_STAGES));
      }
      const int D = step_D(s);
      const int j0 = I.p0 - D;                   // first key of this step
      float corr = 1.f;
      bool rescale_o = false;
      // running-max update shared by both step shapes
      auto update_max = [&](float mx) {
        if (mx > m_ref + kRescaleThreshold || (m_ref == -INFINITY && mx != -INFINITY)) {
          const float m_new = fmaxf(m_ref, mx);
          corr = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - m_new);
          rescale_o = (s > 0) && (m_ref != -INFINITY);
          l *= corr;
          m_ref = m_new;
        }
      };
      if (s < I.s2) {
        // ---------------- half step: 32 keys per thread, relative bias
        const uint32_t sbuf = tmem + lane_base + TM_H + 64u * (uint32_t)(s & 1);
        // the newest chunk this step needs (older ones were awaited before)
        // (chunk c landed: its P stage may be refilled)
        if (s == 0) {
          for (int c = I.c_start; c <= I.c_first && ok; ++c) {
            ok = warp_wait(bar(B_R_FULL + chunk_idx(c) % 3), (chunk_idx(c) / 3) & 1, 14);
            if (ok && leader) mbar_arrive(bar(B_PS_EMPTY + chunk_idx(c) % P_STAGES));
          }
        } else {
          const int c = c_new(s);
          if (c >= I.c_start) {
            ok = warp_wait(bar(B_R_FULL + chunk_idx(c) % 3), (chunk_idx(c) / 3) & 1, 15);
            if (ok && leader) mbar_arrive(bar(B_PS_EMPTY + chunk_idx(c) % P_STAGES));
          }
        }
        if (!ok) break;
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
          if (base >= d_min) tmem_ld32(r_addr(base), w0);
          if (base + 32 >= d_min) tmem_ld32(r_addr(base + 32), w1);
          tmem_wait_ld(sr);
          reg_dep(w0);
          reg_dep(w1);
          // distances below the first computed chunk are not needed: zeros
          // (warp-uniform; only near the start of a decode split's band)
          if (base < d_min) {
#pragma unroll
            for (int i = 0; i < 32; ++i) w0[i] = 0u;
          }
          if (base + 32 < d_min) {
#pragma unroll
            for (int i = 0; i < 32; ++i) w1[i] = 0u;
          }
          // z[63 - i] = window[i]; the thread of lane t needs window[32 + t - u]
          float z[64];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            z[63 - i] = __uint_as_float(w0[i]);
            z[31 - i] = __uint_as_float(w1[i]);
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
            ffma2(x[u], x[u + 1], __uint_as_float(sr[u]), __uint_as_float(sr[u + 1]), qk_over_bias,
                  qk_over_bias, z[u], z[u + 1]);
        } else {
          tmem_wait_ld(sr);
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
          float *zz = z + 18;   // 78 entries
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
            ffma2(x[u], x[u + 1], __uint_as_float(sr[u]), __uint_as_float(sr[u + 1]), qk_over_bias,
                  qk_over_bias, zz[u], zz[u + 1]);
        }
        const bool need_mask =
            (j0 + HN - 1 > I.p0) || (a.window > 0 && j0 < I.p_last - a.window + 1) || (j0 < 0);
        if (need_mask) {
          // visible keys of this row: one range [kmin, kmax] of this thread's keys
          const int jb = j0 + 32 * wg;
          const int kmax = pos - jb;
          const int kmin = max(-jb, a.window > 0 ? pos - a.window + 1 - jb : 0);
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = (i >= kmin && i <= kmax) ? x[i] : -INFINITY;
        }
        // x holds t = |alpha| S + bias; the logit in log2 units is t * cbias
        const float mloc = row_max(x) * cbias;
        const float mo = exchange(mloc, ok);
        if (!ok) break;
        update_max(fmaxf(mloc, mo));
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        uint32_t pk[16];
        l += exp_pack_raw(x, cbias, m_use, pk);
        __syncwarp();
        tmem_st16(sbuf + 16u * wg, pk);   // P (bf16 pairs) over S columns [16 wg, 16 wg + 16)
      } else {
        // ---------------- full step: 64 keys per thread, no bias
        // Each thread also reads the other warpgroup's half of its row to take
        // the full row max itself (bit-identical in both warpgroups), so the
        // two warpgroups never meet.  Once S(s) is read, the MMA issuer may
        // compute S(s+2) into its buffer; P goes to the separate P buffer as
        // soon as PV(s-1) has consumed the previous P.
        const uint32_t sbuf = tmem + lane_base + TM_S + 128u * (uint32_t)(full_idx(s) & 1);
        tc_fence_after();
        uint32_t sr0[32], sr1[32], so[32];
        __syncwarp();
        tmem_ld32(sbuf + 64u * wg, sr0);
        tmem_ld32(sbuf + 64u * wg + 32u, sr1);
        tmem_ld32(sbuf + 64u * (1 - wg), so);
        tmem_wait_ld(sr0);
        reg_dep(sr1);
        reg_dep(so);
        float x[64];   // raw scores; the scale is applied inside the exponent
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = __uint_as_float(sr0[i]);
          x[32 + i] = __uint_as_float(sr1[i]);
        }
        const bool need_mask =
            (j0 + BN - 1 > I.p0) || (a.window > 0 && j0 < I.p_last - a.window + 1) || (j0 < 0);
        // visible keys of this row: one range of key indices; kmin / kmax relative to j0
        const int kmax = pos - j0;
        const int kmin = max(-j0, a.window > 0 ? pos - a.window + 1 - j0 : 0);
        float mo;
        {
          float y[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(so[i]);
          if (need_mask) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int k = 64 * (1 - wg) + i;
              y[i] = (k >= kmin && k <= kmax) ? y[i] : -INFINITY;
            }
          }
          mo = row_max(y);
          __syncwarp();
          tmem_ld32(sbuf + 64u * (1 - wg) + 32u, so);
          tmem_wait_ld(so);
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(so[i]);
          if (need_mask) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int k = 64 * (1 - wg) + 32 + i;
              y[i] = (k >= kmin && k <= kmax) ? y[i] : -INFINITY;
            }
          }
          mo = fmaxf(mo, row_max(y));
        }
        // this thread has read all of S(s): its buffer may take S(s+2)
        tc_fence_before();
        mbar_arrive(bar(B_S_READ + (full_idx(s) & 1)));
        if (need_mask) {
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            const int k = 64 * wg + i;
            x[i] = (k >= kmin && k <= kmax) ? x[i] : -INFINITY;
          }
        }
        update_max(fmaxf(row_max(x), mo) * cqk);
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        uint32_t pk[32];
        l += exp_pack_raw(x, cqk, m_use, pk);
        if (s > I.s2) {
          // this warpgroup's half of PV(s-1) has consumed its half of the P
          // buffer; the second half (issued last) also frees the V stage
          if (!(ok = warp_wait(bar(B_PV_F + 2 * wg + (full_idx(s - 1) & 1)), (full_idx(s - 1) >> 1) & 1, 18)))
            break;
          if (wg == 1 && warp == 8 && lane == 0)
            mbar_arrive(bar(B_V_EMPTY + vslot(step_tile(s - 1)) % V_STAGES));
        }
        tc_fence_after();
        __syncwarp();
        tmem_st32(tmem + lane_base + TM_P + 32u * wg, pk);   // P (bf16 pairs), keys [64 wg, 64 wg + 64)
      }
      // O is only touched when some row of this warp needs a rescale; then
      // PV(s-1) must have landed first.  Otherwise PV(s) simply queues behind
      // PV(s-1) on the tensor core.  Full steps have waited for PV(s-1) above
      // (the first full step: S(s2) was issued after PV(s2-1)).  In the band
      // PV(s-1) is known done when S(s+1) lands (issued after it without
      // waiting for P(s)); where S(s+1) does not exist or waits for P(s) (the
      // switch to full steps), by its own commit.
      // TMEM loads / stores are warp-collective: the whole warp rescales its 32
      // rows when any of them needs it (rows that do not are scaled by 1).
      // Half steps: each warpgroup its half of the O columns (PV(s) waits for
      // both warpgroups' P).  Full steps: warpgroup 0 alone, all 128 columns --
      // the first half of PV(s) is issued as soon as warpgroup 0's P is in and
      // writes every O column, so a rescale by warpgroup 1 could overlap it
      // (both warpgroups take the same rescale decision for a row).
      const bool half = s < I.s2;
      if (__any_sync(0xffffffffu, rescale_o) && (half || wg == 0)) {
        if (half) {
          if (s + 1 >= I.nsteps) ok = warp_wait(bar(B_PV_TAIL), n_tail0 & 1, 16);   // after PV(nsteps - 2)
          else if (s + 1 == I.s2) ok = warp_wait(bar(B_PV_SW), n_sw & 1, 16);       // after PV(s2 - 2)
          else ok = warp_wait(bar(B_S_FULL + step_kind(s + 1)), step_phase(s + 1), 16);
          if (!ok) break;
        } else if (s > I.s2) {
          // both halves of PV(s-1) write every O column: wait for the second
          if (!(ok = warp_wait(bar(B_PV_F + 2 + (full_idx(s - 1) & 1)), (full_idx(s - 1) >> 1) & 1, 16))) break;
        }
        tc_fence_after();
        const float cf = rescale_o ? corr : 1.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (half && c >= 2) break;
          uint32_t r[32];
          const uint32_t oaddr = tmem + lane_base + TM_O + (half ? 64u * wg : 0u) + 32u * c;
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
      if (s < I.s2) mbar_arrive(bar(B_P_FULL + step_kind(s)));
      else mbar_arrive(bar(B_P_HALF + 2 * wg + (full_idx(s) & 1)));
    }
    (void)delta;
    // ---- epilogue.  The next item's q / r rows go in first: its first MMAs
    // (r.P chunks, S) run while this item's output is written.
    const int nsteps_e = I.nsteps, tail_par = n_tail1 & 1, v_last = vslot(I.ntiles - 1) % V_STAGES;
    const int s2_e = (DECODE && WALK) ? I.s2 : 0;
    const int v_band_last = (DECODE && WALK) ? vslot(I.nb_tiles - 1) % V_STAGES : 0;
    const bool valid = a_row < I.nrows;
    const size_t qrow = (size_t)(I.cq + t_row) * a.Hq + h_row;
    // decode with several splits leaves fp32 partials for the combine kernel
    const bool partial = DECODE && a.num_splits > 1;
    const size_t part_row = (size_t)I.split * a.total_q * a.Hq + qrow;
    const size_t lse_at = (size_t)h_row * a.total_q + I.cq + t_row;
    finish_item();
    have = ok && next_item();
    if (have && !q_slot) stage_item();
    if (ok && nsteps_e > 0) ok = warp_wait(bar(B_PV_TAIL + 1), tail_par, 17);
    // PV of the last step has landed: the last tile's V stage is free (the
    // steps release every earlier one, except, in decode, the last half-step
    // tile when exactly one full step follows the band: its release point,
    // the landing of S(s2 + 1), would be a step past the item's end.  A
    // prefill CTA that walks items has band steps only.)
    if (ok && leader && nsteps_e > 0) mbar_arrive(bar(B_V_EMPTY + v_last));
    if constexpr (DECODE && WALK) {
      if (ok && leader && s2_e > 0 && nsteps_e == s2_e + 1) mbar_arrive(bar(B_V_EMPTY + v_band_last));
    }
    float l_other = 0.f;
    // total row sum over both key halves
    if (ok) l_other = exchange(l, ok);
    if (ok) {
      const float lt = l + l_other;
      tc_fence_after();
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float row_lse = lt > 0.f ? (m_ref + __log2f(lt)) * kLn2 : -INFINITY;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        if (nsteps_e > 0) {
          __syncwarp();
          tmem_ld32(tmem + lane_base + TM_O + 64u * wg + 32u * c, r);
          tmem_wait_ld(r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;   // an empty split contributes nothing
        }
        if (valid && partial) {
          float *dst = a.o_part + part_row * kHeadDim + 64 * wg + 32 * c;
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
        if (partial) a.lse_part[part_row] = row_lse;
        else a.lse[lse_at] = row_lse;
      }
    }
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
    for (int t = max(0, issued_k - K_STAGES); t < issued_k; ++t)
      if (t != a.test_skip_k_tile)
        mbar_wait(bar(B_K_FULL + t % K_STAGES), (t / K_STAGES) & 1, &keep_waiting, 2, 400000000ll);
    for (int t = max(0, issued_v - V_STAGES); t < issued_v; ++t)
      mbar_wait(bar(B_V_FULL + t % V_STAGES), (t / V_STAGES) & 1, &keep_waiting, 2, 400000000ll);
    for (int o = max(0, issued_p - P_STAGES); o < issued_p; ++o)
      mbar_wait(bar(B_PS_FULL + o % P_STAGES), (o / P_STAGES) & 1, &keep_waiting, 2, 400000000ll);
    if (issued_rt > 0)
      mbar_wait(bar(B_RT_FULL), (issued_rt - 1) & 1, &keep_waiting, 2, 400000000ll);
  }
  if (warp == 1) {
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
  if (a.rd > 0 && a.E > 0) {
    // P slices are TMA boxes of 64 distances: rel_extent >= 64, rows of 16 bytes
    if (a.rd % 8 != 0 || a.E % 8 != 0 || a.rd > 64 || a.E < HN || !al(a.r) || !al(a.P)) return false;
  }
  if (total_k < BN) return false;   // K/V boxes stay inside the tensor
  return true;
}

namespace {

template <bool DECODE, bool WALK>
cudaError_t launch_tc(const KernelArgs &a, int total_k, dim3 grid, cudaStream_t stream) {
  TcArgs ta;
  ta.a = a;
  ta.has_bias = a.rd > 0 && a.E > 0;
  CUtensorMap mk, mv, mp;
  {
    cuuint64_t dims[3] = {128, (cuuint64_t)a.Hkv, (cuuint64_t)total_k};
    cuuint64_t strides[2] = {256, (cuuint64_t)a.Hkv * 256};
    cuuint32_t box[3] = {64, 1, BN};
    if (!encode(&mk, a.k, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!encode(&mv, a.v, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  if (ta.has_bias) {
    // P [r_dim, E]: box of 64 distances x r_dim channels (x offsets are
    // multiples of 64 elements, i.e. of 128 bytes)
    cuuint64_t dims[2] = {(cuuint64_t)a.E, (cuuint64_t)a.rd};
    cuuint64_t strides[1] = {(cuuint64_t)a.E * 2};
    cuuint32_t box[2] = {(cuuint32_t)HN, (cuuint32_t)a.rd};
    if (!encode(&mp, a.P, 2, dims, strides, box)) return cudaErrorInvalidValue;
  } else {
    mp = mk;   // unused
  }
  // prefill, bias band alone, alpha > 0, r_dim a multiple of 16 (no padding
  // channels): q and r rows by TMA.  q [total_q, Hq, 128] in boxes of 64
  // dims x 128 rows; r [total_q, Hq, r_dim] in one box of 64 channels x 128
  // rows (channels past r_dim read as 0)
  CUtensorMap mq = mk, mr = mk;
  ta.stage_tma = !DECODE && a.band_only && ta.has_bias && a.alpha_log2e > 0.f && a.rd == a.rd_pad &&
                 a.rd <= 64 && a.total_q >= BM;
  if (ta.stage_tma) {
    cuuint64_t dq[3] = {128, (cuuint64_t)a.Hq, (cuuint64_t)a.total_q};
    cuuint64_t sq[2] = {256, (cuuint64_t)a.Hq * 256};
    cuuint32_t bq[3] = {64, 1, BM};
    cuuint64_t dr[3] = {(cuuint64_t)a.rd, (cuuint64_t)a.Hq, (cuuint64_t)a.total_q};
    cuuint64_t sr[2] = {(cuuint64_t)a.rd * 2, (cuuint64_t)a.Hq * a.rd * 2};
    cuuint32_t br[3] = {64, 1, BM};
    if (!encode(&mq, a.q, 3, dq, sq, bq) || !encode(&mr, a.r, 3, dr, sr, br)) ta.stage_tma = 0;
  }
  static std::atomic<bool> attr_set[kMaxDevicesAttr];
  cudaError_t e = set_max_smem_once(reinterpret_cast<const void *>(relattn_fwd_tc_kernel<DECODE, WALK>),
                                    (int)SMEM_BYTES, attr_set);
  if (e != cudaSuccess) return e;
  relattn_fwd_tc_kernel<DECODE, WALK><<<grid, NTHREADS, SMEM_BYTES, stream>>>(ta, mk, mv, mp, mq, mr);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const KernelArgs &a, int total_k, cudaStream_t stream) {
  // one item per CTA, except for the bias band alone: then one CTA per SM
  // walks the items (no per-CTA set-up, and the next item's tiles load while
  // the current one finishes)
  const long items = (long)a.q_tiles * a.Hq * a.batch;
  if (items <= 0) return cudaSuccess;
  const long ctas = a.band_only && a.sms > 0 && items > a.sms ? (long)a.sms : items;
  if (ctas > 0x7fffffffL) return cudaErrorInvalidValue;
  return launch_tc<false, true>(a, total_k, dim3((unsigned)ctas, 1, 1), stream);
}

cudaError_t launch_decode_tc(const KernelArgs &a, int total_k, cudaStream_t stream) {
  // at most one CTA per SM, each walking items (the longest first): the next
  // item's tiles load while the current one finishes, and the set-up is paid
  // once per SM instead of once per (sequence, split, kv head, row block)
  // (items that fit in one wave keep one CTA each, without the item loop's
  // bookkeeping: about 3.5 % faster on a 1M-key decode of 152 items)
  const long items = (long)a.num_splits * a.Hkv * a.row_blocks * a.batch;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffL) return cudaErrorInvalidValue;
  if (a.sms <= 0 || items <= a.sms)
    return launch_tc<true, false>(a, total_k, dim3(a.num_splits, a.Hkv * a.row_blocks, a.batch), stream);
  return launch_tc<true, true>(a, total_k, dim3((unsigned)a.sms, 1, 1), stream);
}

}  // namespace relattn
