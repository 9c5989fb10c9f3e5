// decode_tc.cu -- split-KV decode of relative attention for items of few query
// rows (at most 16: one token of a GQA group of up to 16 heads, or a couple of
// tokens of a smaller group), on 5th-generation tensor cores with the keys
// along the MMA's M dimension.
//
// Same computation as the definition on the page "SGLang and Miles Add Day-0
// Support for Inkling", section "Attention with Relative Positional
// Embedding": x(i,j) = s(i) (alpha q_i.k_j + [0 <= i-j < E] r_i . P[:, i-j]),
// softmax over the visible keys, PV; the keys of a sequence are cut into
// splits whose normalised partials the LSE combine merges (page "vLLM Day-0
// support for TML Inkling", paragraph on FA4 with sheared bias, num_splits).
//
// A decode item is (split, sequence, kv head): its rows are the (token,
// head-in-group) pairs of one kv head -- 8 rows for one token of a GQA-8
// group -- and it streams the split's keys in 128-key tiles.  With so few rows
// both products are computed transposed, with 16 rows as the MMA's N:
// S^T = K Q^T (the tile's 128 keys along M, i.e. TMEM lanes) and
// O^T += V^T P^T (the 128 dims along M), so the tensor core and the softmax
// only touch real rows (the rows-along-M decode of fwd_tc.cu spends 128 lanes
// on them).  Each softmax thread owns one key: it scales its 16 scores, adds
// the relative bias of band tiles and masks edge tiles; the per-row maximum
// over the tile's keys is a transposed warp reduction (lane l ends with row
// l % 16) plus a four-warp exchange; lane l decides row l's running max,
// which the lanes receive by shuffles; then p = 2^(x - m), written to shared
// memory as the B operand of the PV product.  Each key-thread keeps its share
// of every row's sum; the shares are reduced once per item.
//
// Two softmax warpgroups take the item's tiles in turn (tile G of the CTA's
// walk goes to warpgroup G % 2), each with its own running max and sum, its
// own P buffer and its own O^T accumulator: a warpgroup has two tile periods
// for each of its tiles, so the softmax hides behind the copies and the
// tensor core.  At the end of the item the two partial results are merged
// like two splits (the max of the two running maxima, each side rescaled).
//
// Relative bias, R = r . P, from one of two sources; a band tile reads R at
// (row, p_row - j) per (key, row), all sixteen loads issued before any is used.
//   In the kernel (bf16 K / V, r_dim a multiple of 8, E <= 1152): P^T sits in
//   tensor memory for the whole launch (lane = distance, loaded once per CTA
//   by the softmax warps), and for each item that reaches the band the score
//   issuer computes R^T = P^T r^T of its rows on the tensor core (M = 128
//   distances, N = 16 rows, one 128-distance block at a time) right after the
//   item's q and r rows land; each softmax warpgroup copies it at the item's
//   start into its own slot in the workspace (fp32 [distance][row]), from
//   which its band tiles read.  The slot is private to the warpgroup, so only
//   the warpgroup's own barrier orders the copy before the reads.
//   Otherwise (MXFP8 K / V, other shapes): R for every decode row and
//   distance below E is computed beforehand (relattn_decode_rel_kernel, fp32
//   [row][E] in the workspace) and the decode is launched as its programmatic
//   dependent.
//
// Work split: with several splits (and at most 64 sequences) the walk is
// stream-K: the (sequence, kv head) units' tiles are laid end to end and CTA
// c takes the range [c C, (c + 1) C), C = ceil(total / CTAs) (at least a
// bound that keeps every unit within num_splits pieces); each piece of a unit
// writes its partial into split slot c - (first CTA of the unit), the unit's
// first piece marks the slots no piece fills as empty, and the combine merges
// them.  Every CTA then streams the same number of tiles.  Otherwise each CTA
// walks a fixed share of the (split, sequence, kv head) items in a
// longest-first order.
//
// Warps (11; one CTA per SM):
//   warp 0      TMA producer (one thread): the item's q rows (a box of group
//               heads x tokens), then K and V tiles (rings of 2-4 stages); the
//               rings run on across items
//   warp 1      TMEM allocator, score MMA issuer (the warp runs the issue
//               code, an elected lane issues): S^T(G) into the buffer of
//               warpgroup G % 2
//   warp 10     P V MMA issuer (likewise): O^T += V^T P^T of tile G into
//               warpgroup G % 2's accumulator once its P is written
//   warps 2-5   softmax warpgroup 0 (even tiles), warps 6-9 warpgroup 1 (odd
//               tiles): thread = key of the tile (TMEM lane 32 (warp % 4) +
//               lane) for the scores, = dim of O^T for the rescale and merge
//
// Tensor memory (64 columns; 512 with the in-kernel R): S^T of warpgroup b at
// 16 b, O^T of warpgroup b at 32 + 16 b; then P^T (32 columns per 128
// distances) and the current item's R^T (16 per 128 distances).
// Shared memory: the two P buffers (16 rows x 128 keys, 4 KB each), the q
// rows of two items (4 KB each: the next item's load while the current one
// runs) and their r rows (2 KB each), K and V rings, the merge buffer
// (warpgroup 1's O^T, 8 KB), per-warpgroup row constants and exchange buffers.
//
// Every wait is bounded; a timeout raises the CTA's abort flag and records the
// wait site in the device error word; the CTA drains its copies and MMAs,
// frees its tensor memory and exits.
#include <cudaTypedefs.h>

#include "launch.h"
#include "mxfp8.cuh"
#include "tc_common.cuh"

namespace relattn {
namespace {

using namespace tc;

constexpr int KT = 128;                    // keys per tile (TMEM lanes of S^T)
constexpr int NR = kFewRows;               // rows per item at most (the MMAs' N)
static_assert(NR == 16, "one 16-column chunk of S^T");
constexpr int MAXST = 4;                   // K or V ring stages at most (the layouts pick their own)
constexpr int NTHR = 352;                  // 11 warps (roles below)
constexpr int PV_WARP = 10;
constexpr float kRescale = 8.f;            // log2 units

constexpr uint32_t BOX = 16384;            // 128 rows of 128 bytes (64 bf16 dims or 128 fp8 dims), 128B swizzle
constexpr uint32_t HALF16 = NR * 128;      // 16 rows of 128 bytes: 2 KB
// per warpgroup: row constants and exchange buffers
constexpr uint32_t WG_ROWC = 0;                       // float4 [NR]: scale, bias scale, position, output row
constexpr uint32_t WG_RSC = WG_ROWC + NR * 16;        // float [NR]: the scales, packed
constexpr uint32_t WG_MREF = WG_RSC + NR * 4;         // float [2][NR]: running max by tile parity
constexpr uint32_t WG_XMAX = WG_MREF + 2 * NR * 4;    // float [2][NR][4]: tile max per warp
constexpr uint32_t WG_AUX = WG_XMAX + 2 * NR * 16;    // float [NR][4]: row sums per warp
constexpr uint32_t WG_BYTES = WG_AUX + NR * 16;
// work order (batch <= kOrd): per sequence its full / partial split counts,
// their prefix sums, the partial splits by size, the count of partials, and
// the sequence offsets (cu_seqlens_q / _k, read once per CTA)
constexpr int kOrd = 64;
constexpr int ORD_NF = 0, ORD_REM = kOrd, ORD_PF = 2 * kOrd, ORD_PZ = 3 * kOrd + 1,
              ORD_PTAB = 4 * kOrd + 2, ORD_NP = 5 * kOrd + 2, ORD_CQ = 5 * kOrd + 4,
              ORD_CK = 6 * kOrd + 5, ORD_INTS = 7 * kOrd + 6;
enum {
  B_Q_FULL = 0, B_Q_EMPTY = B_Q_FULL + 2, B_K_FULL = B_Q_EMPTY + 2, B_K_EMPTY = B_K_FULL + MAXST, B_V_FULL = B_K_EMPTY + MAXST,
  B_V_EMPTY = B_V_FULL + MAXST, B_S_FULL = B_V_EMPTY + MAXST, B_S_FREE = B_S_FULL + 2,
  B_P_FULL = B_S_FREE + 2, B_PV_DONE = B_P_FULL + 2, B_XCH = B_PV_DONE + 2, B_M_FULL = B_XCH + 2,
  B_M_FREE = B_M_FULL + 1, B_DRAIN = B_M_FREE + 1, B_DRAIN_PV = B_DRAIN + 1, B_R_FULL = B_DRAIN_PV + 1,
  B_R_FREE = B_R_FULL + 1, B_PT_READY = B_R_FREE + 1, B_PT_SMEM_FULL = B_PT_READY + 1,
  B_PT_SMEM_FREE = B_PT_SMEM_FULL + 1, B_COUNT = B_PT_SMEM_FREE + 1
};
// In-kernel R (bf16 kernel): tensor-memory columns past S and O.  P^T takes 32
// columns (64 bf16 channels) per 128 distances, the R of one item 16 columns
// (one per row) per 128 distances.
constexpr uint32_t TM_PT = 64;
constexpr int kRelTmemCols = 512;
constexpr int kRelMaxBlocks = 8;   // P staged once in the V ring: 8 x (128 distances x 64 channels) bf16

// Tensor- and shared-memory layout of the bf16 kernel (F8 = false) and of the
// MXFP8 one (K / V stored as E4M3 codes with one E8M0 scale per 32 dims, q
// quantised the same way per item, V dequantised to bf16 per tile).
//   TMEM: S^T of warpgroup b at TM_S + SCOLS b (fp8: four 16-column blocks, one
//   per 32 head dims, scaled in the softmax); O^T of warpgroup b at TM_O + 16 b.
//   SMEM: the two P buffers (4 KB each), the q rows of two items (bf16: 4 KB,
//   fp8: 2 KB each), K and V rings, (fp8) each warpgroup's bf16 V tile, the
//   merge buffer, (fp8) the q scales of two items, per-warpgroup buffers, the
//   work order, barriers.
template <bool F8>
struct Lay {
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t SCOLS = F8 ? 4 * NR : NR;
  static constexpr uint32_t TM_O = 2 * SCOLS;
  static constexpr uint32_t TMEM_COLS = F8 ? 256 : 64;
  static constexpr uint32_t KTILE = F8 ? BOX : 2 * BOX;       // bytes of one K (or V) stage
  static constexpr uint32_t QBUF = F8 ? HALF16 : 2 * HALF16;  // bytes of one item's q rows
  static constexpr uint32_t SM_P = 0;
  static constexpr uint32_t SM_Q = SM_P + 4 * HALF16;
  static constexpr uint32_t SM_R = SM_Q + 4 * HALF16;         // bf16: the r rows of two items (2 KB each)
  static constexpr uint32_t SM_K = SM_R + (F8 ? 0 : 2 * HALF16);
  // ring stages: K is released right after its score MMA, V only after its
  // P V MMA (bf16) or its dequantisation (fp8), so V holds its stages longer
  // and gets more of them; at the loaded memory's ~2.5 us latency the bytes in
  // flight, not the bandwidth, set the pace
  static constexpr int KST = F8 ? 4 : 2, VST = 4;
  static constexpr uint32_t SM_V = SM_K + KST * KTILE;
  static constexpr uint32_t SM_VB = SM_V + VST * KTILE;       // fp8: bf16 V of warpgroup b at + 2 BOX b
  static constexpr uint32_t SM_MB = SM_VB + (F8 ? 4 * BOX : 0);   // float [NR][128]: warpgroup 1's O^T; m, l [NR]
  static constexpr uint32_t SM_QSC = SM_MB + NR * 128 * 4 + 2 * NR * 4;  // fp8: float [2][NR][4]
  static constexpr uint32_t SM_WG = SM_QSC + (F8 ? 2 * NR * 16 : 0);
  static constexpr uint32_t SM_ORD = SM_WG + 2 * WG_BYTES;
  static constexpr uint32_t SM_BAR = SM_ORD + ORD_INTS * 4;
  static constexpr uint32_t SM_TMEM_SLOT = SM_BAR + B_COUNT * 8;
  static constexpr uint32_t SM_ABORT = SM_TMEM_SLOT + 8;
  static constexpr uint32_t SM_TOTAL = SM_ABORT + 8;
  static constexpr uint32_t SMEM_BYTES = SM_TOTAL + 1024;      // + alignment slack
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(SM_K % 1024 == 0 && SM_VB % 1024 == 0 && SM_WG % 16 == 0 && SM_QSC % 16 == 0,
                "alignment");
};

struct DecArgs {
  KernelArgs a;
  const uint32_t *kscale, *vscale;   // MXFP8: E8M0 scale bytes of each (row, kv head), 4 per word
  int kv_rows;                       // rows of the K / V tensors
  int has_bias;
  // where the relative bias comes from: 1 = R of every decode row computed
  // beforehand (a.rdec, [total_q * Hq][E]); 2 = computed in the kernel, per
  // item with band tiles, into this CTA's slots (rslot)
  int rel_mode;
  // stream-K walk (several splits, at most kOrd sequences): CTA c takes tiles
  // [c C, (c + 1) C) of the (sequence, kv head) units laid end to end, with
  // C = max(c_min, ceil(total tiles / CTAs)); c_min caps a unit's pieces at
  // num_splits
  int streamk, c_min;
  int nt_e;          // 128-distance blocks of E
  int rs;            // floats per distance in a slot: the item's rows, rounded up to 4
  int r_bytes;       // bytes of the item's r box
  float *rslot;      // per (CTA, softmax warpgroup): R^T [nt_e * 128][rs] fp32
  int q_bytes;       // bytes of the item's q box pair
  int n_items;
};

// Reduction over the warp's 32 lanes of each of the 16 per-lane values, left
// transposed: lane l gets the result for value l % 16.  Halving stages over
// the lane bits that select the value (a lane keeps half of its values and
// trades the other half with its partner): 16 shuffles, independent within a
// stage, instead of 16 full-warp reductions in a chain.
template <bool MAX>
__device__ __forceinline__ float transpose_reduce(const float (&v)[NR], int lane) {
  float a[NR];
#pragma unroll
  for (int i = 0; i < NR; ++i) a[i] = v[i];
#pragma unroll
  for (int w = NR / 2; w >= 1; w >>= 1) {
    const bool hi = (lane & w) != 0;
#pragma unroll
    for (int k = 0; k < w; ++k) {
      const float send = hi ? a[k] : a[k + w];
      const float keep = hi ? a[k + w] : a[k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, w);
      a[k] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  const float o = __shfl_xor_sync(0xffffffffu, a[0], 16);
  return MAX ? fmaxf(a[0], o) : a[0] + o;
}

struct Item {
  int b, g, sp, cq, ck, nrows, p0, p_last, kbeg, ntiles;
  int np;   // stream-K: the pieces of the item's (sequence, kv head) unit
};

template <bool F8>
__global__ void __launch_bounds__(NTHR, 1)
relattn_decode_tc_kernel(const __grid_constant__ DecArgs da,
                         const __grid_constant__ CUtensorMap map_q,
                         const __grid_constant__ CUtensorMap map_k,
                         const __grid_constant__ CUtensorMap map_v,
                         const __grid_constant__ CUtensorMap map_r,
                         const __grid_constant__ CUtensorMap map_p) {
  using L = Lay<F8>;
  const KernelArgs &a = da.a;
  extern __shared__ uint8_t smem_raw[];
  // 1024-aligned base, kept as an offset into the shared array so that every
  // access below stays a shared-memory access (32-bit addresses)
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_addr(smem);
  auto bar = [&](int i) { return sb + L::SM_BAR + 8u * i; };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::SM_ABORT);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ------------------------------------------------------------ work items
  // An item is a (sequence, split) pair times Hkv kv heads.  With at most
  // kOrd sequences the pairs are ordered full splits first, then the partial
  // last splits by size, then the empty ones, and slot idx of the walk maps to
  // a position in that order by rounds of gridDim.x slots, every other full
  // round reversed (a snake): the longest items start first and the rounds
  // even out.  Every role derives the same order from the same tables.
  // Otherwise the plain order: pair = split * batch + sequence.
  Item I{};
  int *ord = reinterpret_cast<int *>(smem + L::SM_ORD);
  const bool sorted = a.batch <= kOrd;
  const bool sk = da.streamk != 0 && sorted;
  auto load_item_into = [&](int idx, Item &it) -> int {   // 1 work, 0 nothing, -1 inconsistent lengths
    int q, u;
    int t_lo = 0, t_hi = 0;
    if (sk) {
      // piece idx of this CTA's tile range: unit u_a + idx, the part of its
      // tiles inside [R0, R1)
      const int C = ord[ORD_NP], T = ord[ORD_PF + a.batch];
      const int uu = ord[ORD_NP + 1] + idx;
      it.b = uu / a.Hkv;
      u = uu - it.b * a.Hkv;
      const int U = ord[ORD_NF + it.b], P = ord[ORD_PF + it.b] + u * U;
      const int R0 = (int)blockIdx.x * C, R1 = min(R0 + C, T);
      t_lo = max(R0, P) - P;
      t_hi = min(R1, P + U) - P;
      it.sp = (int)blockIdx.x - P / C;
      it.np = U > 0 ? (P + U - 1) / C - P / C + 1 : 0;
      // (a unit never has more pieces than split slots: c_min sees to that)
      if (it.sp < 0 || it.np > a.num_splits) return -1;
    } else if (sorted) {
      const int Gd = gridDim.x, r = idx / Gd, c = idx - r * Gd;
      const int pos = ((r & 1) && (r + 1) * Gd <= da.n_items) ? r * Gd + (Gd - 1 - c) : idx;
      q = pos / a.Hkv;
      u = pos - q * a.Hkv;
      const int F = ord[ORD_PF + a.batch], NP = ord[ORD_NP];
      if (q < F || q >= F + NP) {
        const int base = q < F ? ORD_PF : ORD_PZ, qq = q < F ? q : q - F - NP;
        int b = 0;                                       // last b with prefix[b] <= qq
        for (int i = 1; i < a.batch; ++i) b = ord[base + i] <= qq ? i : b;
        it.b = b;
        it.sp = q < F ? qq - ord[ORD_PF + b]
                     : ord[ORD_NF + b] + (ord[ORD_REM + b] > 0 ? 1 : 0) + (qq - ord[ORD_PZ + b]);
      } else {
        it.b = ord[ORD_PTAB + (q - F)];
        it.sp = ord[ORD_NF + it.b];
      }
    } else {
      q = idx / a.Hkv;
      u = idx - q * a.Hkv;
      it.b = q % a.batch;
      it.sp = q / a.batch;
    }
    it.g = u;
    const int *cq_t = sorted ? ord + ORD_CQ : a.cu_q, *ck_t = sorted ? ord + ORD_CK : a.cu_k;
    it.cq = cq_t[it.b];
    it.ck = ck_t[it.b];
    const int Lq = cq_t[it.b + 1] - it.cq, Lk = ck_t[it.b + 1] - it.ck;
    // (rows past total_q would index outputs and R out of bounds)
    if (Lq < 0 || Lk < Lq || Lq > a.max_q || Lk > a.max_k || it.cq < 0 || it.cq + Lq > a.total_q) return -1;
    if (Lq == 0) return 0;
    it.nrows = Lq * a.group;
    it.p0 = Lk - Lq;
    it.p_last = it.p0 + Lq - 1;
    const int j_lo = a.window > 0 ? max(0, it.p0 - a.window + 1) : 0;
    const int kbase = j_lo & ~(KT - 1);
    if (sk) {
      it.kbeg = kbase + KT * t_lo;
      it.ntiles = max(0, t_hi - t_lo);
      return 1;
    }
    it.kbeg = kbase + it.sp * a.split_chunk;
    const int kend = min(it.p_last + 1, it.kbeg + a.split_chunk);
    it.ntiles = kend > it.kbeg ? (kend - it.kbeg + KT - 1) / KT : 0;
    it.np = a.num_splits;
    return 1;
  };
  auto load_item = [&](int idx) -> int { return load_item_into(idx, I); };
  const int n_items = da.n_items;
  // in-kernel R: tile t of an item is a band tile iff t >= first_band(it)
  // (its oldest key is within E of the item's first row); an item computes R
  // iff it has a band tile
  const bool rel_tc = !F8 && da.rel_mode == 2;
  auto first_band = [&](const Item &it) -> int {
    const int x = it.p0 - it.kbeg - (KT - 1) - a.E;
    return x < 0 ? 0 : x / KT + 1;
  };
  auto band_item = [&](const Item &it) -> bool { return rel_tc && first_band(it) < it.ntiles; };
  // the 128-distance blocks an item's band tiles read: its distances run
  // from p0 - (last key of its tiles) to p_last - (first key), clipped to E
  auto r_lo = [&](const Item &it) -> int { return max(0, it.p0 - (it.kbeg + KT * it.ntiles - 1)) / KT; };
  auto r_hi = [&](const Item &it) -> int { return min(da.nt_e - 1, (it.p_last - it.kbeg) / KT); };
  const uint32_t tmem_cols = rel_tc ? (uint32_t)kRelTmemCols : L::TMEM_COLS;
  const uint32_t TM_RS = TM_PT + 32u * (uint32_t)da.nt_e;   // R of the current item

  // ------------------------------------------------------------ set-up
  // q and the P buffers start as zeros: rows past an item's real ones then
  // score 0 instead of whatever the memory held
  for (int i = tid; i < (int)(L::SM_K - L::SM_P) / 16; i += NTHR)
    *reinterpret_cast<uint4 *>(smem + L::SM_P + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_Q_FULL + i), 1);
      mbar_init(bar(B_Q_EMPTY + i), F8 ? 1 + 256 : 1);   // fp8: + the softmax threads (q scales)
    }
    for (int i = 0; i < MAXST; ++i) {
      mbar_init(bar(B_K_FULL + i), 1);
      mbar_init(bar(B_K_EMPTY + i), 1);
      mbar_init(bar(B_V_FULL + i), 1);
      mbar_init(bar(B_V_EMPTY + i), F8 ? 128 : 1);   // fp8: the dequantising warpgroup's threads
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_S_FULL + i), 1);
      mbar_init(bar(B_S_FREE + i), 128);
      mbar_init(bar(B_P_FULL + i), 128);
      mbar_init(bar(B_PV_DONE + i), 1);
      mbar_init(bar(B_XCH + i), 128);
    }
    mbar_init(bar(B_M_FULL), 128);
    mbar_init(bar(B_M_FREE), 128);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_DRAIN_PV), 1);
    mbar_init(bar(B_R_FULL), 1);
    mbar_init(bar(B_R_FREE), 256);
    mbar_init(bar(B_PT_READY), 256);
    mbar_init(bar(B_PT_SMEM_FULL), 1);
    mbar_init(bar(B_PT_SMEM_FREE), 256);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + L::SM_TMEM_SLOT, tmem_cols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map_q);
    prefetch_tmap(&map_k);
    prefetch_tmap(&map_v);
    if (rel_tc) {
      prefetch_tmap(&map_r);
      prefetch_tmap(&map_p);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (sorted) {
    // the work order: each sequence's keys from the aligned start of its
    // window, cut into splits of split_chunk keys
    const int b = tid;
    if (b < a.batch) {
      const int cq = a.cu_q[b], ck = a.cu_k[b];
      const int cq1 = a.cu_q[b + 1], ck1 = a.cu_k[b + 1];
      ord[ORD_CQ + b + 1] = cq1;
      ord[ORD_CK + b + 1] = ck1;
      if (b == 0) {
        ord[ORD_CQ] = cq;
        ord[ORD_CK] = ck;
      }
      const int Lq = cq1 - cq, Lk = ck1 - ck;
      long vis = 0;
      if (Lq > 0 && Lk >= Lq) {
        const int p0 = Lk - Lq, p_last = p0 + Lq - 1;
        const int j_lo = a.window > 0 ? max(0, p0 - a.window + 1) : 0;
        vis = (long)p_last + 1 - (j_lo & ~(KT - 1));
      }
      const long nf = min((long)a.num_splits, vis / a.split_chunk);
      // (stream-K: the unit's tiles instead)
      ord[ORD_NF + b] = sk ? (int)((vis + KT - 1) / KT) : (int)nf;
      ord[ORD_REM + b] = nf < a.num_splits ? (int)(vis - nf * a.split_chunk) : 0;
    }
    __syncthreads();
    if (sk) {
      // stream-K: tiles before each sequence's units, the CTA's range and
      // its first unit and piece count
      if (tid == 0) {
        int t = 0;
        for (int i = 0; i < a.batch; ++i) {
          ord[ORD_PF + i] = t;
          t += a.Hkv * ord[ORD_NF + i];
        }
        ord[ORD_PF + a.batch] = t;
        const int C = max(da.c_min, (t + (int)gridDim.x - 1) / (int)gridDim.x);
        const int R0 = (int)blockIdx.x * C, R1 = min(R0 + C, t);
        auto unit_of = [&](int tile) {   // the unit holding tile (tile < t)
          int b = 0;
          while (b + 1 < a.batch && ord[ORD_PF + b + 1] <= tile) ++b;
          return b * a.Hkv + (tile - ord[ORD_PF + b]) / ord[ORD_NF + b];
        };
        const int ua = R0 < t ? unit_of(R0) : 0;
        ord[ORD_NP] = C;
        ord[ORD_NP + 1] = ua;
        ord[ORD_PZ] = R0 < t ? unit_of(R1 - 1) - ua + 1 : 0;
      }
    } else if (tid == 0) {
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
    if (b < a.batch && ord[ORD_REM + b] > 0) {   // rank among the partial splits: larger first
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
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::SM_TMEM_SLOT);
  // this CTA's walk: idx = w0, w0 + wS, ... below wN (stream-K: its pieces in
  // order; else every gridDim.x-th slot of the order)
  const int w0 = sk ? 0 : (int)blockIdx.x, wS = sk ? 1 : (int)gridDim.x, wN = sk ? ord[ORD_PZ] : n_items;
  // the combine after this kernel may launch (it waits for every CTA's partials)
  asm volatile("griddepcontrol.launch_dependents;");
  // the producer's copies, drained if the CTA gives up
  int issued_q = 0, issued_k = 0, issued_v = 0;
  bool issued_pt = false;

  if (warp == 0) {
    // ====================================================== TMA producer
    // Two cursors over the CTA's tiles: the K copies run ahead as soon as a K
    // stage is free (after its score MMA), the V copies as soon as a V stage
    // is (after its P V MMA, or for fp8 after its dequantisation), so a late V
    // stage never holds back the next K tile.  Each item's q rows go first
    // (bf16: a TMA box; fp8: the whole warp quantises them).  The loop is
    // warp-uniform: lane 0 probes the barriers and issues the copies, the
    // decisions are broadcast.
    Item ik{}, iv{};
    int kidx = w0 - wS, vidx = kidx, kt = 0, vt = 0;
    int GK = 0, GV = 0, n_q = 0;
    auto next_item = [&](int &idx, Item &it) -> bool {
      for (idx += wS; idx < wN; idx += wS) {
        const int li = load_item_into(idx, it);
        if (li < 0 && lane == 0 && &it == &ik) atomicOr(a.err, kDevErrSeqlens);
        if (li > 0 && it.ntiles > 0) return true;
      }
      return false;
    };
    auto ready = [&](uint32_t br, uint32_t parity) -> bool {
      const bool r = lane == 0 ? mbar_test_wait(br, parity) : false;
      return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
    };
    // the pool row of tile t of item it (paged K / V: a 128-aligned tile inside one page)
    auto tile_row = [&](const Item &it, int t) -> int {
      const int p = it.kbeg + KT * t;
      if (a.block_table == nullptr) return it.ck + p;
      const int pg = a.block_table[(size_t)it.b * a.max_pages + p / a.page_size];
      if (pg < 0 || pg >= a.num_pages) {
        atomicOr(a.err, kDevErrSeqlens);
        return -KT;   // reads zeros
      }
      return pg * a.page_size + p % a.page_size;
    };
    bool k_live = next_item(kidx, ik), v_live = next_item(vidx, iv), q_due = k_live;
    long long idle_since = -1;
    // in-kernel R: P [r_dim][E] into the (still empty) V ring, 128 distances
    // x r_dim channels per box; the V copies start once the softmax warps
    // have moved it into tensor memory
    bool pt_free = !rel_tc;
    if (rel_tc) {
      if (lane == 0) {
        const uint32_t box = 256u * (uint32_t)a.rd;
        mbar_arrive_expect_tx(bar(B_PT_SMEM_FULL), box * (uint32_t)da.nt_e);
        for (int u = 0; u < da.nt_e; ++u)
          tma_load_2d(sb + L::SM_V + box * (uint32_t)u, &map_p, KT * u, 0, bar(B_PT_SMEM_FULL));
      }
      issued_pt = true;
    }
    for (;;) {
      // (lane 0's view of the abort flag, so the whole warp leaves together)
      const bool quit = __shfl_sync(0xffffffffu, (lane == 0 && *abort_flag) ? 1 : 0, 0) != 0;
      if (!(k_live || v_live) || quit) break;
      bool moved = false;
      if (k_live && q_due) {
        const int qb = n_q & 1;
        if (n_q < 2 || ready(bar(B_Q_EMPTY + qb), ((n_q >> 1) - 1) & 1)) {
          if constexpr (F8) {
            // the item's q rows, MXFP8 per 32 dims, into the K-major operand of
            // S^T; each (row, block) scale times the row's logit scale
            uint8_t *q8 = smem + L::SM_Q + qb * L::QBUF;
            float *qsc = reinterpret_cast<float *>(smem + L::SM_QSC) + qb * NR * 4;
            for (int pr = lane; pr < NR * 4; pr += 32) {
              const int r = pr >> 2, blk = pr & 3;
              uint32_t c[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
              float sc = 0.f;
              if (r < ik.nrows) {
                const int tau = r / a.group, hg = r - tau * a.group;
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    a.q + ((size_t)(ik.cq + tau) * a.Hq + ik.g * a.group + hg) * kHeadDim + 32 * blk);
                int e;
                quantize_block32(src, c, e);
                sc = a.alpha_log2e * log_scale(ik.p0 + tau, a.inv_ln_base) * pow2i(e);
              }
              // codes of dims 32 blk .. 32 blk + 31 of row r: 16-byte chunks 2 blk, 2 blk + 1
              *reinterpret_cast<uint4 *>(q8 + r * 128 + (((2 * blk) ^ (r & 7)) << 4)) =
                  make_uint4(c[0], c[1], c[2], c[3]);
              *reinterpret_cast<uint4 *>(q8 + r * 128 + (((2 * blk + 1) ^ (r & 7)) << 4)) =
                  make_uint4(c[4], c[5], c[6], c[7]);
              qsc[r * 4 + blk] = sc;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_Q_FULL + qb));
          } else if (lane == 0) {
            // the item's q rows: [tokens][group heads][128 dims] as two 2 KB halves of 64 dims;
            // with in-kernel R, an item with band tiles also brings its r rows
            // ([tokens][group heads][64 channels], channels past r_dim read as 0)
            const bool rb = band_item(ik);
            mbar_arrive_expect_tx(bar(B_Q_FULL + qb), (uint32_t)(da.q_bytes + (rb ? da.r_bytes : 0)));
            tma_load_3d(sb + L::SM_Q + qb * L::QBUF, &map_q, 0, ik.g * a.group, ik.cq, bar(B_Q_FULL + qb));
            tma_load_3d(sb + L::SM_Q + qb * L::QBUF + HALF16, &map_q, 64, ik.g * a.group, ik.cq,
                        bar(B_Q_FULL + qb));
            if (rb) tma_load_3d(sb + L::SM_R + qb * HALF16, &map_r, 0, ik.g * a.group, ik.cq, bar(B_Q_FULL + qb));
          }
          issued_q = ++n_q;
          q_due = false;
          moved = true;
        }
      } else if (k_live) {
        const int st = GK % L::KST;
        if (GK < L::KST || ready(bar(B_K_EMPTY + st), ((GK / L::KST) - 1) & 1)) {
          if (lane == 0 && GK != a.test_skip_k_tile) {   // (test hook: a skipped tile is never loaded)
            const int row = tile_row(ik, kt);
            mbar_arrive_expect_tx(bar(B_K_FULL + st), L::KTILE);
            tma_load_3d(sb + L::SM_K + st * L::KTILE, &map_k, 0, ik.g, row, bar(B_K_FULL + st));
            if constexpr (!F8)
              tma_load_3d(sb + L::SM_K + st * L::KTILE + BOX, &map_k, 64, ik.g, row, bar(B_K_FULL + st));
          }
          issued_k = ++GK;
          if (++kt == ik.ntiles) {
            kt = 0;
            k_live = next_item(kidx, ik);
            q_due = k_live;
          }
          moved = true;
        }
      }
      if (!pt_free) pt_free = ready(bar(B_PT_SMEM_FREE), 0);
      if (v_live && GV < GK && pt_free) {
        const int st = GV % L::VST;
        if (GV < L::VST || ready(bar(B_V_EMPTY + st), ((GV / L::VST) - 1) & 1)) {
          if (lane == 0) {
            const int row = tile_row(iv, vt);
            mbar_arrive_expect_tx(bar(B_V_FULL + st), L::KTILE);
            tma_load_3d(sb + L::SM_V + st * L::KTILE, &map_v, 0, iv.g, row, bar(B_V_FULL + st));
            if constexpr (!F8)
              tma_load_3d(sb + L::SM_V + st * L::KTILE + BOX, &map_v, 64, iv.g, row, bar(B_V_FULL + st));
          }
          issued_v = ++GV;
          if (++vt == iv.ntiles) {
            vt = 0;
            v_live = next_item(vidx, iv);
          }
          moved = true;
        }
      }
      // bounded: a stretch without progress longer than about a second gives
      // up (lane 0's clock decides for the warp)
      if (moved) {
        idle_since = -1;
      } else {
        __nanosleep(64);   // back off: the softmax warps share this sub-partition
        const long long now = clock64();
        if (idle_since < 0) idle_since = now;
        const bool give_up = __shfl_sync(0xffffffffu, (now - idle_since > 2000000000ll) ? 1 : 0, 0) != 0;
        if (give_up) {
          if (lane == 0) *abort_flag = 2;
          break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ====================================================== score MMA issuer
    // The whole warp runs the issue code (descriptors stay warp-uniform); each
    // MMA and commit is issued by one elected lane.
    {
      const uint32_t id_s = idesc_bf16_f32(KT, NR, 0, 0);    // S^T = K Q^T: K (keys x dims), q rows, both K-major
      // descriptor bases; k-step k of a 128-wide K dimension: +2 per 32 bytes
      // inside a 128-byte row, the second 64-wide half at +16 KB in a K tile
      // and at +2 KB in the 16-row q and P operands (fp8: the K codes hold
      // all 128 dims in one 128-byte row, 32 dims per E4M3 k-step); V^T:
      // dims along M in two 64-dim boxes 16 KB apart, 16 keys (+2 KB) per k-step
      const uint64_t qd0 = smem_desc_sw128(sb + L::SM_Q, 16, 1024);
      const uint64_t kd0 = smem_desc_sw128(sb + L::SM_K, 16, 1024);
      const uint32_t id_s8 = idesc_e4m3_f32(KT, NR);
      auto koff = [](int k) -> uint64_t { return (uint64_t)((k < 4) ? 2 * k : (BOX >> 4) + 2 * (k - 4)); };
      auto hoff = [](int k) -> uint64_t { return (uint64_t)((k < 4) ? 2 * k : (HALF16 >> 4) + 2 * (k - 4)); };
      // in-kernel R: R^T[d][row] = P^T[d] . r[row] per 128-distance block
      // (P^T in TMEM as the A operand, the item's r rows K-major in shared memory)
      const uint64_t rd0 = smem_desc_sw128(sb + L::SM_R, 16, 1024);
      const int r_ksteps = a.rd_pad / 16;
      int T = 0, n_it = 0, n_rel = 0;
      bool ok = true;
      for (int idx = w0; idx < wN && ok; idx += wS) {
        if (load_item(idx) <= 0 || I.ntiles == 0) continue;
        const int qb = n_it & 1;
        if (!(ok = mbar_wait_warp(bar(B_Q_FULL + qb), (n_it >> 1) & 1, abort_flag, 6))) break;
        const uint64_t qd = qd0 + (uint64_t)((qb * L::QBUF) >> 4);
        // in-kernel R of a band item, one 128-distance block at a time ahead
        // of the score MMAs of the tiles before the band, so that the last
        // block goes in before S of the tile before the first band tile (or
        // all of them before S(0) when the band starts at once)
        const bool rb = band_item(I);
        const int t_b = rb ? first_band(I) : I.ntiles;
        const int u_lo = rb ? r_lo(I) : 0, n_u = rb ? r_hi(I) - u_lo + 1 : 0;
        int r_done = 0;   // blocks issued: u_lo .. u_lo + r_done - 1
        auto issue_r = [&](int upto) -> bool {
          if (r_done >= upto) return true;
          if (r_done == 0) {
            // P^T is in TMEM (once per CTA); the previous item's R has been read out
            if (n_rel == 0 && !mbar_wait_warp(bar(B_PT_READY), 0, abort_flag, 21)) return false;
            if (n_rel > 0 && !mbar_wait_warp(bar(B_R_FREE), (n_rel - 1) & 1, abort_flag, 22)) return false;
            tc_fence_after();
          }
          const uint64_t rdesc = rd0 + (uint64_t)((qb * HALF16) >> 4);
          for (; r_done < upto; ++r_done) {
            const uint32_t u = (uint32_t)(u_lo + r_done);
            const uint32_t d = tmem + TM_RS + 16u * u, pa = tmem + TM_PT + 32u * u;
            mma_ts_e<0>(d, pa, rdesc, id_s);
            for (int k = 1; k < r_ksteps; ++k) mma_ts_e<1>(d, pa + 8u * (uint32_t)k, rdesc + 2 * k, id_s);
          }
          if (r_done == n_u) {
            mma_commit_e(bar(B_R_FULL));
            ++n_rel;
          }
          return true;
        };
        for (int t = 0; t < I.ntiles && ok; ++t) {
          const int G = T + t, b = G & 1, st = G % L::KST;
          if (rb && t <= t_b && !(ok = issue_r(min(n_u, max(0, n_u - (t_b - 1 - t)))))) break;
          if (G >= 2 && !(ok = mbar_wait_warp(bar(B_S_FREE + b), ((G >> 1) - 1) & 1, abort_flag, 7))) break;
          if (!(ok = mbar_wait_warp(bar(B_K_FULL + st), (G / L::KST) & 1, abort_flag, 8))) break;
          tc_fence_after();
          const uint64_t kd = kd0 + (uint64_t)((st * L::KTILE) >> 4);
          const uint32_t d = tmem + L::TM_S + L::SCOLS * (uint32_t)b;
          if constexpr (F8) {
            // one product per 32-dim block, each into its own 16 columns (the
            // block scales differ, so the softmax combines them)
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_f8_e<0>(d + 16u * k, kd + 2 * k, qd + 2 * k, id_s8);
          } else {
            mma_ss_e<0>(d, kd + koff(0), qd + hoff(0), id_s);
#pragma unroll
            for (int k = 1; k < 8; ++k) mma_ss_e<1>(d, kd + koff(k), qd + hoff(k), id_s);
          }
          mma_commit_e(bar(B_S_FULL + b));
          mma_commit_e(bar(B_K_EMPTY + st));
          if (t == I.ntiles - 1) mma_commit_e(bar(B_Q_EMPTY + qb));   // the item's q rows are read
        }
        T += I.ntiles;
        ++n_it;
      }
      // drain: every MMA issued above has finished before TMEM is released
      mma_commit_e(bar(B_DRAIN));
      volatile int keep_waiting = 0;
      mbar_wait(bar(B_DRAIN), 0, &keep_waiting, 9, 400000000ll);
    }
    __syncwarp();
  } else if (warp == PV_WARP) {
    // ====================================================== PV issuer
    // A second issuing thread for the P V products, so the score MMAs of the
    // next tiles and the P V MMA of a finished tile do not wait on one
    // another's waits (each issuing lane's commits track only its own MMAs).
    // The whole warp runs it; an elected lane issues.
    {
      const uint32_t id_o = idesc_bf16_f32(128, NR, 1, 0);   // O^T += V^T P^T: V^T dims-contiguous, P K-major
      const uint64_t pd0 = smem_desc_sw128(sb + L::SM_P, 16, 1024);
      const uint64_t vd0 = smem_desc_sw128(sb + (F8 ? L::SM_VB : L::SM_V), BOX, 1024);
      auto hoff = [](int k) -> uint64_t { return (uint64_t)((k < 4) ? 2 * k : (HALF16 >> 4) + 2 * (k - 4)); };
      int T = 0;
      bool ok = true;
      for (int idx = w0; idx < wN && ok; idx += wS) {
        if (load_item(idx) <= 0 || I.ntiles == 0) continue;
        for (int t = 0; t < I.ntiles && ok; ++t) {
          // O^T of warpgroup G % 2 (+)= V(G)^T P(G)^T; the warpgroup's first tile of the item overwrites
          const int G = T + t, st = G % L::VST, b = G & 1;
          if (!(ok = mbar_wait_warp(bar(B_P_FULL + b), (G >> 1) & 1, abort_flag, 4))) break;
          // (fp8: P_FULL also says the warpgroup's bf16 V tile is written)
          if (!F8 && !(ok = mbar_wait_warp(bar(B_V_FULL + st), (G / L::VST) & 1, abort_flag, 5))) break;
          tc_fence_after();
          const uint64_t vd = vd0 + (uint64_t)(((F8 ? b * 2 * BOX : st * L::KTILE)) >> 4);
          const uint64_t pd = pd0 + (uint64_t)((b * 2 * HALF16) >> 4);
          const uint32_t o = tmem + L::TM_O + 16u * (uint32_t)b;
          if (t < 2) mma_ss_e<0>(o, vd + 0, pd + hoff(0), id_o);
          else mma_ss_e<1>(o, vd + 0, pd + hoff(0), id_o);
#pragma unroll
          for (int k = 1; k < 8; ++k) mma_ss_e<1>(o, vd + 128 * k, pd + hoff(k), id_o);
          mma_commit_e(bar(B_PV_DONE + b));
          if (!F8) mma_commit_e(bar(B_V_EMPTY + st));
        }
        T += I.ntiles;
      }
      mma_commit_e(bar(B_DRAIN_PV));
      volatile int keep_waiting = 0;
      mbar_wait(bar(B_DRAIN_PV), 0, &keep_waiting, 9, 400000000ll);
    }
    __syncwarp();
  } else {
    // ======================================================== softmax
    const int wg = (warp - 2) >> 2;              // warpgroup: tiles G with G % 2 == wg
    const int wq = warp & 3;                     // TMEM lane quarter of this warp
    const int key = 32 * wq + lane;              // this thread's key of the tile / dim of O^T
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    const bool row_owner = wq == 0;              // lanes 0..15 of this warp: rows 0..15
    const int r_own = lane & (NR - 1);           // the row this lane decides (lanes 16-31 repeat)
    uint8_t *wgs = smem + L::SM_WG + wg * WG_BYTES;
    float4 *rowc = reinterpret_cast<float4 *>(wgs + WG_ROWC);
    float *rsc = reinterpret_cast<float *>(wgs + WG_RSC);
    float *mref = reinterpret_cast<float *>(wgs + WG_MREF);
    float *xmax = reinterpret_cast<float *>(wgs + WG_XMAX);
    float *aux = reinterpret_cast<float *>(wgs + WG_AUX);
    float *mbuf = reinterpret_cast<float *>(smem + L::SM_MB);          // [NR][128]
    float *mbuf_m = mbuf + NR * 128, *mbuf_l = mbuf_m + NR;
    const uint32_t s_col = tmem + lane_base + L::TM_S + L::SCOLS * (uint32_t)wg;
    const uint32_t o_col = tmem + lane_base + L::TM_O + 16u * (uint32_t)wg;
    const uint32_t p_buf = L::SM_P + (uint32_t)wg * 2 * HALF16;
    const bool has_bias = da.has_bias != 0;
    const bool partial = a.num_splits > 1;
    auto warp_wait = [&](uint32_t br, uint32_t parity, int site) -> bool {
      const bool r = mbar_wait(br, parity, abort_flag, site);
      return __all_sync(0xffffffffu, r);
    };
    int n_xch = 0, n_merge = 0, n_rel = 0;
    bool r_ready = false;
    bool ok = true;
    // the warpgroup's 128 threads meet
    auto xch_barrier = [&]() -> bool {
      mbar_arrive(bar(B_XCH + wg));
      return warp_wait(bar(B_XCH + wg), (n_xch++) & 1, 10);
    };
    // in-kernel R: this warpgroup's slot, R^T [nt_e * 128 distances][rs rows]
    const uint32_t rslot_off = rel_tc ? ((uint32_t)blockIdx.x * 2u + (uint32_t)wg) * (uint32_t)(da.nt_e * 128 * da.rs) : 0u;
    if (rel_tc) {
      // P^T into TMEM, once per CTA, from the copy of P the producer put in
      // the V ring ([r_dim][128] bf16 per block of 128 distances; distances
      // past E read as 0): lane = distance 128 u + key of block u (warpgroup
      // wg takes the blocks u = wg mod 2), channels as bf16 pairs over 32
      // columns, zero past r_dim.  Then the V ring is the producer's again.
      ok = warp_wait(bar(B_PT_SMEM_FULL), 0, 24);
      if (ok) {
        for (int u = wg; u < da.nt_e; u += 2) {
          const unsigned short *src =
              reinterpret_cast<const unsigned short *>(smem + L::SM_V + 256u * (uint32_t)a.rd * (uint32_t)u) + key;
          uint32_t w[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const uint32_t lo = 2 * c < a.rd ? (uint32_t)src[(2 * c) * 128] : 0u;
            const uint32_t hi = 2 * c + 1 < a.rd ? (uint32_t)src[(2 * c + 1) * 128] : 0u;
            w[c] = lo | (hi << 16);
          }
          __syncwarp();
          tmem_st32(tmem + lane_base + TM_PT + 32u * (uint32_t)u, w);
        }
        mbar_arrive(bar(B_PT_SMEM_FREE));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(B_PT_READY));
      }
    }
    // in-kernel R: this warpgroup's copy of the current item's R into its slot
    // (thread = distance 128 u + key, its rs rows as 16-byte stores), then the
    // warpgroup meets so that every thread's stores precede every band read
    auto extract_r = [&]() -> bool {
      if (!warp_wait(bar(B_R_FULL), n_rel & 1, 23)) return false;
      tc_fence_after();
      // (four columns per load: the copy runs inside the tile loop, where
      // the row sums and scores hold most registers)
      const int u_end = r_hi(I);
      for (int u = r_lo(I); u <= u_end; ++u) {
        float4 *dst = reinterpret_cast<float4 *>(da.rslot + rslot_off + (uint32_t)((128 * u + key) * da.rs));
        for (int q4 = 0; 4 * q4 < da.rs; ++q4) {
          uint32_t v[4];
          tmem_ld4(tmem + lane_base + TM_RS + 16u * (uint32_t)u + 4u * (uint32_t)q4, v);
          tmem_wait_ld(v);
          dst[q4] = make_float4(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]),
                                __uint_as_float(v[3]));
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_R_FREE));
      return xch_barrier();
    };
    int T = 0;
    for (int idx = w0; idx < wN && ok; idx += wS) {
      const int li = load_item(idx);
      if (li <= 0) continue;
      const int nrows = I.nrows;
      // ---- row constants (thread = row), once the warpgroup is done with the previous item's
      if (!(ok = xch_barrier())) break;
      if (key < NR) {
        const int r = key;
        float4 v = make_float4(0.f, 0.f, __int_as_float(0x7fffffff), __int_as_float(-1));
        if (r < nrows) {
          const int tau = r / a.group, hg = r - tau * a.group;
          const int pos = I.p0 + tau;
          const float s = log_scale(pos, a.inv_ln_base);
          v = make_float4(a.alpha_log2e * s, kLog2e * s, __int_as_float(pos),
                          __int_as_float((I.cq + tau) * a.Hq + I.g * a.group + hg));
        }
        rowc[r] = v;
        rsc[r] = v.x;
        mref[r] = -INFINITY;
        mref[NR + r] = -INFINITY;
      }
      if (!(ok = xch_barrier())) break;
      if (I.ntiles == 0) {
        // an empty split of a multi-split decode: its partial contributes nothing
        if (wg == 0 && partial && key < nrows) {
          const size_t qrow = (size_t)__float_as_int(rowc[key].w);
          float *dst = a.o_part + ((size_t)I.sp * a.total_q * a.Hq + qrow) * kHeadDim;
          for (int i = 0; i < kHeadDim; i += 4) *reinterpret_cast<float4 *>(dst + i) = make_float4(0.f, 0.f, 0.f, 0.f);
          a.lse_part[(size_t)I.sp * a.total_q * a.Hq + qrow] = -INFINITY;
        }
        continue;
      }
      float lp[NR];                              // this key's share of each row's sum
#pragma unroll
      for (int i = 0; i < NR; ++i) lp[i] = 0.f;
      int tl = 0;                                // this warpgroup's tiles of the item so far
      // in-kernel R: this warpgroup copies the item's R just before its first
      // band tile t_w -- at the end of its tile t_w - 2, or at the top of t_w
      // when that is its first tile of the item
      // (copy_at: t_w while the copy is due, else -4)
      int copy_at = -4;
      if (band_item(I)) {
        const int t_b = first_band(I);
        copy_at = t_b + ((t_b - ((wg - T) & 1)) & 1);
      }
      for (int t = (wg - T) & 1; t < I.ntiles && ok; t += 2, ++tl) {
        const int G = T + t;
        const int j0 = I.kbeg + KT * t, j = j0 + key;
        const bool band = has_bias && (I.p_last - j0 >= 0) && (I.p0 - (j0 + KT - 1) < a.E);
        const bool edge = (j0 + KT - 1 > I.p0) || (a.window > 0 && j0 < I.p_last - a.window + 1);
        if (t == copy_at) {
          if (!(ok = extract_r())) break;
          copy_at = -4;
        }
        // band tiles: R[row][p_row - j] for this key, every load issued before
        // the S wait (an index outside the band reads R[0] and is discarded)
        float rbias[NR];
        if (band && !rel_tc && !r_ready) {
          // launched as a programmatic dependent of the R kernel: its rows are
          // complete and visible past this point
          asm volatile("griddepcontrol.wait;" ::: "memory");
          r_ready = true;
        }
        if (band && rel_tc && (a.group & 3) == 0) {
          // rows in fours of one token: one 16-byte load per four rows
#pragma unroll
          for (int q4 = 0; q4 < NR / 4; ++q4) {
            const int dd = __float_as_int(rowc[4 * q4].z) - j;
            const bool in = dd >= 0 && dd < a.E && 4 * q4 < da.rs;
            const float4 rv =
                *reinterpret_cast<const float4 *>(da.rslot + rslot_off + (in ? (uint32_t)(dd * da.rs + 4 * q4) : 0u));
            rbias[4 * q4] = in ? rv.x * rowc[4 * q4].y : 0.f;
            rbias[4 * q4 + 1] = in ? rv.y * rowc[4 * q4 + 1].y : 0.f;
            rbias[4 * q4 + 2] = in ? rv.z * rowc[4 * q4 + 2].y : 0.f;
            rbias[4 * q4 + 3] = in ? rv.w * rowc[4 * q4 + 3].y : 0.f;
          }
        } else if (band && rel_tc) {
#pragma unroll
          for (int i = 0; i < NR; ++i) {
            const float4 rc = rowc[i];
            const int dd = __float_as_int(rc.z) - j;
            const bool in = dd >= 0 && dd < a.E && i < da.rs;
            const float rv = da.rslot[rslot_off + (in ? (uint32_t)(dd * da.rs + i) : 0u)];
            rbias[i] = in ? rv * rc.y : 0.f;
          }
        } else if (band) {
#pragma unroll
          for (int i = 0; i < NR; ++i) {
            const float4 rc = rowc[i];
            const int dd = __float_as_int(rc.z) - j;
            const bool in = dd >= 0 && dd < a.E;
            const size_t at = in ? (size_t)__float_as_int(rc.w) * a.E + dd : 0;
            const float rv = a.rdec[at];
            rbias[i] = in ? rv * rc.y : 0.f;
          }
        }
        // fp8: this key's K and V block scales (4 E8M0 bytes each; rows past
        // the tensor, which the copies fill with zeros, take 2^0)
        uint32_t ksw = 0x7F7F7F7Fu, vsw = 0x7F7F7F7Fu;
        if constexpr (F8) {
          const int kr = I.ck + j;
          if (kr < da.kv_rows) {
            ksw = da.kscale[(size_t)kr * a.Hkv + I.g];
            vsw = da.vscale[(size_t)kr * a.Hkv + I.g];
          }
        }
        if (!(ok = warp_wait(bar(B_S_FULL + wg), (G >> 1) & 1, 12))) break;
        tc_fence_after();
        float y[NR];
        if constexpr (F8) {
          // S^T of the four 32-dim blocks; y = sum_b S_b * (row scale x q block
          // scale) * k block scale
          const float kf0 = pow2i((int)(ksw & 0xFFu) - 127), kf1 = pow2i((int)((ksw >> 8) & 0xFFu) - 127);
          const float kf2 = pow2i((int)((ksw >> 16) & 0xFFu) - 127), kf3 = pow2i((int)(ksw >> 24) - 127);
          const float4 *qs4 = reinterpret_cast<const float4 *>(smem + L::SM_QSC) + (n_merge & 1) * NR;
          uint32_t r[32];
          tmem_ld32(s_col, r);   // blocks 0 and 1
          tmem_wait_ld(r);
#pragma unroll
          for (int i = 0; i < NR; ++i) {
            const float4 qs = qs4[i];
            y[i] = fmaf(__uint_as_float(r[16 + i]), qs.y * kf1, __uint_as_float(r[i]) * (qs.x * kf0));
          }
          tmem_ld32(s_col + 32, r);   // blocks 2 and 3
          tmem_wait_ld(r);
#pragma unroll
          for (int i = 0; i < NR; ++i) {
            const float4 qs = qs4[i];
            y[i] = fmaf(__uint_as_float(r[16 + i]), qs.w * kf3, fmaf(__uint_as_float(r[i]), qs.z * kf2, y[i]));
          }
        } else {
          uint32_t r[16];
          tmem_ld16(s_col, r);
          tmem_wait_ld(r);
#pragma unroll
          for (int i = 0; i < NR; ++i) y[i] = __uint_as_float(r[i]);
        }
        tc_fence_before();
        mbar_arrive(bar(B_S_FREE + wg));          // this thread has read S^T(G)
        // scale (packed row scales: 4 broadcast vector loads), bias, masks
        if constexpr (!F8) {
          const float4 *sc4 = reinterpret_cast<const float4 *>(rsc);
#pragma unroll
          for (int q4 = 0; q4 < NR / 4; ++q4) {
            const float4 sv = sc4[q4];
            y[4 * q4] *= sv.x;
            y[4 * q4 + 1] *= sv.y;
            y[4 * q4 + 2] *= sv.z;
            y[4 * q4 + 3] *= sv.w;
          }
        }
        if (band) {
#pragma unroll
          for (int i = 0; i < NR; ++i) y[i] += rbias[i];
        }
        if (edge) {
#pragma unroll
          for (int i = 0; i < NR; ++i) {
            const int pos = __float_as_int(rowc[i].z);
            if (!(j <= pos && (a.window <= 0 || j > pos - a.window))) y[i] = -INFINITY;
          }
        }
        // the tile's per-row maximum over this warp's keys (lane l: row l % 16),
        // then over the four warps
        float *xm = xmax + (tl & 1) * (NR * 4);
        {
          const float mx = transpose_reduce<true>(y, lane);
          if (lane < NR) xm[4 * lane + wq] = mx;
        }
        if (!(ok = xch_barrier())) break;
        // lane l decides row l % 16's new running max (every warp decides the
        // same); the lanes receive each row's by shuffles; p = 2^(y - m); this
        // key's share of each row's sum, rescaled with the row's max
        const float *mo = mref + (tl & 1) * NR;
        float *mn = mref + ((tl + 1) & 1) * NR;
        const float4 w4 = reinterpret_cast<const float4 *>(xm)[r_own];
        const float mx = fmaxf(fmaxf(w4.x, w4.y), fmaxf(w4.z, w4.w));
        const float m_old = mo[r_own];
        const bool upd = mx > m_old + kRescale || (m_old == -INFINITY && mx != -INFINITY);
        const float m_new = upd ? fmaxf(m_old, mx) : m_old;
        const float corr = !upd ? 1.f : (m_old == -INFINITY ? 0.f : fast_exp2(m_old - m_new));
        const bool any_rescale = __any_sync(0xffffffffu, upd && tl > 0 && m_old != -INFINITY);
        const bool any_upd = __any_sync(0xffffffffu, upd);
        if (row_owner && lane < NR) mn[r_own] = m_new;
        const float mb = m_new == -INFINITY ? 0.f : m_new;
        if (any_upd) {
#pragma unroll
          for (int i = 0; i < NR; ++i) {
            const float p = fast_exp2(y[i] - __shfl_sync(0xffffffffu, mb, i));
            lp[i] = fmaf(lp[i], __shfl_sync(0xffffffffu, corr, i), p);
            y[i] = p;
          }
        } else {
#pragma unroll
          for (int i = 0; i < NR; ++i) {
            const float p = fast_exp2(y[i] - __shfl_sync(0xffffffffu, mb, i));
            lp[i] += p;
            y[i] = p;
          }
        }
        // this warpgroup's P buffer and O^T are free once its previous tile's
        // PV (tile G - 2: of this item, or of an earlier one) has landed
        if (G >= 2 && !(ok = warp_wait(bar(B_PV_DONE + wg), ((G - 2) >> 1) & 1, 13))) break;
        tc_fence_after();
        if (any_rescale) {
          // O^T[dim][row] times the row's factor (the whole warpgroup: thread = dim)
          uint32_t r[16];
          tmem_ld16(o_col, r);
          tmem_wait_ld(r);
#pragma unroll
          for (int i = 0; i < NR; ++i)
            r[i] = __float_as_uint(__uint_as_float(r[i]) * __shfl_sync(0xffffffffu, corr, i));
          tmem_st16(o_col, r);
          tmem_wait_st();
        }
        if constexpr (F8) {
          // this key's V codes (one 128-byte row of the stage) dequantised into
          // the warpgroup's bf16 V tile: dims 0-63 in the first 128-byte-swizzled
          // box, 64-127 in the second; then the stage is free for the next copy
          const int st = G % L::VST;
          if (!(ok = warp_wait(bar(B_V_FULL + st), (G / L::VST) & 1, 19))) break;
          const uint8_t *v8 = smem + L::SM_V + st * L::KTILE + key * 128;
          uint8_t *vb = smem + L::SM_VB + wg * 2 * BOX + key * 128;
          const uint32_t sw = (uint32_t)(key & 7);
#pragma unroll
          for (int c = 0; c < 8; ++c) {   // 16 dims per 16-byte chunk of codes
            const uint4 w = *reinterpret_cast<const uint4 *>(v8 + ((c ^ sw) << 4));
            const float s = pow2i((int)((vsw >> (8 * (c >> 1))) & 0xFFu) - 127);
            uint32_t o[8];
            dequant4_bf16(w.x, s, o[0], o[1]);
            dequant4_bf16(w.y, s, o[2], o[3]);
            dequant4_bf16(w.z, s, o[4], o[5]);
            dequant4_bf16(w.w, s, o[6], o[7]);
            uint8_t *box = vb + (c >> 2) * BOX;
            *reinterpret_cast<uint4 *>(box + ((((2 * c) & 7) ^ sw) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4 *>(box + ((((2 * c + 1) & 7) ^ sw) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
          mbar_arrive(bar(B_V_EMPTY + st));
        }
        // P[row][key] (bf16) into the 128-byte-swizzled K-major B operand:
        // keys 0-63 in the first 2 KB half, 64-127 in the second
        {
          const uint32_t kb = p_buf + (uint32_t)(key >> 6) * HALF16 + (uint32_t)((key & 7) << 1);
          const uint32_t kc = (uint32_t)((key & 63) >> 3);
#pragma unroll
          for (int i = 0; i < NR; ++i)
            *reinterpret_cast<__nv_bfloat16 *>(smem + kb + (uint32_t)i * 128u +
                                               ((kc ^ ((uint32_t)i & 7u)) << 4)) = __float2bfloat16_rn(y[i]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(B_P_FULL + wg));
        if (t + 2 == copy_at) {
          if (!(ok = extract_r())) break;
          copy_at = -4;
        }
      }
      if (!ok) break;
      // ---- this warpgroup's row sums and max; its O^T once its last PV has landed
      const int ntl = tl;
      {
        const float sum = transpose_reduce<false>(lp, lane);
        if (lane < NR) aux[4 * lane + wq] = sum;
      }
      if (!(ok = xch_barrier())) break;
      if (ntl > 0) {
        const int G_last = T + ((wg - T) & 1) + 2 * (ntl - 1);
        if (!(ok = warp_wait(bar(B_PV_DONE + wg), (G_last >> 1) & 1, 14))) break;
      }
      tc_fence_after();
      float o[NR];
      {
        uint32_t r[16];
        if (ntl > 0) {
          tmem_ld16(o_col, r);
          tmem_wait_ld(r);
        }
#pragma unroll
        for (int i = 0; i < NR; ++i) o[i] = ntl > 0 ? __uint_as_float(r[i]) : 0.f;
      }
      const float *m_fin = mref + (ntl & 1) * NR;
      if (wg == 1) {
        // ---- warpgroup 1 hands its O^T, max and sums to warpgroup 0
        if (n_merge > 0 && !(ok = warp_wait(bar(B_M_FREE), (n_merge - 1) & 1, 16))) break;
#pragma unroll
        for (int i = 0; i < NR; ++i) mbuf[i * 128 + key] = o[i];
        if (row_owner && lane < NR) {
          const float4 s4 = reinterpret_cast<const float4 *>(aux)[lane];
          mbuf_m[lane] = m_fin[lane];
          mbuf_l[lane] = (s4.x + s4.y) + (s4.z + s4.w);
        }
        mbar_arrive(bar(B_M_FULL));
      } else {
        // ---- warpgroup 0 merges the two halves and writes the rows
        if (!(ok = warp_wait(bar(B_M_FULL), n_merge & 1, 17))) break;
        // thread = dim; row i: m = max(m0, m1), each side scaled by 2^(m_side - m)
        float lrow = 0.f, mrow = -INFINITY;   // lane i (< 16): row i's sum and max, for the lse
#pragma unroll
        for (int i = 0; i < NR; ++i) {
          const float m0 = m_fin[i], m1 = mbuf_m[i];
          const float4 s4 = reinterpret_cast<const float4 *>(aux)[i];
          const float l0 = (s4.x + s4.y) + (s4.z + s4.w), l1 = mbuf_l[i];
          const float m = fmaxf(m0, m1);
          const float f0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - m);
          const float f1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - m);
          const float l = l0 * f0 + l1 * f1;
          const float inv = l > 0.f ? 1.f / l : 0.f;
          const float o1 = mbuf[i * 128 + key];
          o[i] = ((f0 > 0.f ? o[i] * f0 : 0.f) + (f1 > 0.f ? o1 * f1 : 0.f)) * inv;
          if (lane == i) {
            lrow = l;
            mrow = m;
          }
        }
        mbar_arrive(bar(B_M_FREE));
#pragma unroll
        for (int i = 0; i < NR; ++i) {
          if (i >= nrows) break;
          const size_t qrow = (size_t)__float_as_int(rowc[i].w);
          if (partial)
            a.o_part[((size_t)I.sp * a.total_q * a.Hq + qrow) * kHeadDim + key] = o[i];
          else
            a.out[qrow * kHeadDim + key] = __float2bfloat16_rn(o[i]);
        }
        if (row_owner && lane < nrows) {
          const float row_lse = (lrow > 0.f && mrow != -INFINITY) ? (mrow + __log2f(lrow)) * kLn2 : -INFINITY;
          const size_t qrow = (size_t)__float_as_int(rowc[lane].w);
          if (partial) {
            // (stream-K: the unit's first piece marks the split slots no piece
            // of the unit fills as empty)
            if (I.sp == 0)
              for (int s2 = I.np; s2 < a.num_splits; ++s2)
                a.lse_part[(size_t)s2 * a.total_q * a.Hq + qrow] = -INFINITY;
            a.lse_part[(size_t)I.sp * a.total_q * a.Hq + qrow] = row_lse;
          } else {
            const size_t t_row = qrow / a.Hq, h_row = qrow - t_row * a.Hq;
            a.lse[h_row * a.total_q + t_row] = row_lse;
          }
        }
      }
      if constexpr (F8) mbar_arrive(bar(B_Q_EMPTY + (n_merge & 1)));   // the item's q scales are read
      if (band_item(I)) {
        // a warpgroup without a band tile in the item releases its R here,
        // after the merge hand-off: the other warpgroup's release for the
        // previous item is in by then, so the arrivals of two items never mix.
        // It still waits for this item's R first, so that every warpgroup
        // takes every phase of R_FULL in turn (a parity wait that skipped a
        // phase could pass on the one before)
        if (copy_at >= 0) {
          if (!(ok = warp_wait(bar(B_R_FULL), n_rel & 1, 25))) break;
          tc_fence_before();
          mbar_arrive(bar(B_R_FREE));
        }
        ++n_rel;
      }
      ++n_merge;
      T += I.ntiles;
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
    if (issued_pt) mbar_wait(bar(B_PT_SMEM_FULL), 0, &keep_waiting, 15, 400000000ll);
    for (int n = max(0, issued_q - 2); n < issued_q; ++n)
      mbar_wait(bar(B_Q_FULL + (n & 1)), (n >> 1) & 1, &keep_waiting, 15, 400000000ll);
    for (int G = max(0, issued_k - L::KST); G < issued_k; ++G)
      if (G != a.test_skip_k_tile)
        mbar_wait(bar(B_K_FULL + G % L::KST), (G / L::KST) & 1, &keep_waiting, 15, 400000000ll);
    for (int G = max(0, issued_v - L::VST); G < issued_v; ++G)
      mbar_wait(bar(B_V_FULL + G % L::VST), (G / L::VST) & 1, &keep_waiting, 15, 400000000ll);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// R = r . P for every decode row (t, h) and distance d < E, fp32
// [total_q * Hq][E]: a CTA takes 16 rows and 256 distances, a thread one
// distance for the 16 rows.  The CTA's slice of P (r_dim x 256 bf16) is first
// staged in shared memory with 16-byte loads (scalar ones when E is not a
// multiple of 8), all in flight together; the r rows are broadcast from
// shared memory (zero past r_dim, and P's rows past r_dim up to the next
// multiple of 4 are zeroed).
constexpr int RR = 16, RD = 256;
__global__ void __launch_bounds__(RD) relattn_decode_rel_kernel(const KernelArgs a, float *R) {
  // the decode kernel may launch now: it waits for these rows before its first band tile
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ __align__(16) float rs[RR][64];
  __shared__ __align__(16) __nv_bfloat16 ps[64][RD];
  const int tid = threadIdx.x;
  const long rows = (long)a.total_q * a.Hq;
  const long row0 = (long)blockIdx.x * RR;
  const int d0 = blockIdx.y * RD, nd = min(RD, a.E - d0);
  const int rd4 = (a.rd + 3) & ~3;
  if ((a.E & 7) == 0 && (reinterpret_cast<uintptr_t>(a.P) & 15u) == 0) {
    for (int k = tid; k < a.rd * (RD / 8); k += RD) {
      const int c = k / (RD / 8), j = (k % (RD / 8)) * 8;
      if (j < nd)
        *reinterpret_cast<uint4 *>(&ps[c][j]) =
            *reinterpret_cast<const uint4 *>(a.P + (size_t)c * a.E + d0 + j);
    }
  } else {
    for (int k = tid; k < a.rd * RD; k += RD) {
      const int c = k / RD, j = k % RD;
      if (j < nd) ps[c][j] = a.P[(size_t)c * a.E + d0 + j];
    }
  }
  for (int k = a.rd * RD + tid; k < rd4 * RD; k += RD) ps[k / RD][k % RD] = __float2bfloat16_rn(0.f);
  for (int i = tid; i < RR * 64; i += RD) {
    const int rr = i >> 6, c = i & 63;
    rs[rr][c] = (row0 + rr < rows && c < a.rd) ? __bfloat162float(a.r[(row0 + rr) * a.rd + c]) : 0.f;
  }
  __syncthreads();
  if (tid >= nd) return;
  float acc[RR];
#pragma unroll
  for (int i = 0; i < RR; ++i) acc[i] = 0.f;
  for (int c = 0; c < rd4; c += 4) {
    const float p0 = __bfloat162float(ps[c][tid]), p1 = __bfloat162float(ps[c + 1][tid]);
    const float p2 = __bfloat162float(ps[c + 2][tid]), p3 = __bfloat162float(ps[c + 3][tid]);
#pragma unroll
    for (int i = 0; i < RR; ++i) {
      const float4 r4 = *reinterpret_cast<const float4 *>(&rs[i][c]);
      acc[i] = fmaf(r4.x, p0, acc[i]);
      acc[i] = fmaf(r4.y, p1, acc[i]);
      acc[i] = fmaf(r4.z, p2, acc[i]);
      acc[i] = fmaf(r4.w, p3, acc[i]);
    }
  }
  const int d = d0 + tid;
#pragma unroll
  for (int i = 0; i < RR; ++i)
    if (row0 + i < rows) R[(row0 + i) * a.E + d] = acc[i];
}

// With pdl, launch as a programmatic dependent of the kernel before it on the
// stream, which must be the decode-row R kernel: the CTAs start as soon as it
// lets them, and only band tiles wait for its rows.  Otherwise an ordinary
// stream-ordered launch (the kernel before it may be anything).
template <typename K>
cudaError_t launch_decode_kernel(K kernel, int grid, uint32_t smem, cudaStream_t stream, const DecArgs &da,
                                 const CUtensorMap &m0, const CUtensorMap &m1, const CUtensorMap &m2,
                                 const CUtensorMap &m3, const CUtensorMap &m4, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(NTHR);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? &attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, da, m0, m1, m2, m3, m4);
}

// R = r . P of the decode rows before the decode kernel (rel_mode 1)
cudaError_t launch_decode_rel(const KernelArgs &a, cudaStream_t stream) {
  const long rrows = (long)a.total_q * a.Hq;
  dim3 g((unsigned)((rrows + RR - 1) / RR), (unsigned)((a.E + RD - 1) / RD));
  relattn_decode_rel_kernel<<<g, RD, 0, stream>>>(a, const_cast<float *>(a.rdec));
  return cudaGetLastError();
}

// CTAs of a few-row decode launch (one per SM at most)
long decode_grid(const KernelArgs &a, long items) { return std::min<long>(items, a.sms > 0 ? a.sms : items); }

// The walk: stream-K when the keys are cut into several splits (and the
// sequences fit the work-order tables).  A unit (sequence, kv head) holds at
// most U = ceil(num_splits * split_chunk / 128) tiles, and a unit of U tiles
// meets at most ceil(U / C) + 1 ranges of C tiles, so C >= U / (num_splits - 1)
// keeps its pieces within the num_splits partial slots.
void set_walk(const KernelArgs &a, DecArgs &da) {
  da.streamk = (a.num_splits > 1 && a.batch <= kOrd && a.sms > 0) ? 1 : 0;
  da.c_min = 0;
  if (da.streamk) {
    const long umax = ((long)a.num_splits * a.split_chunk + KT - 1) / KT;
    da.c_min = (int)std::max<long>(1, (umax + a.num_splits - 2) / (a.num_splits - 1));
  }
}
// stream-K: one CTA per SM (the ranges even out the work); else one per item
// up to the SM count
int walk_grid(const KernelArgs &a, const DecArgs &da, long items) {
  return da.streamk ? a.sms : (int)decode_grid(a, items);
}

PFN_cuTensorMapEncodeTiled_v12000 dec_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return nullptr;
  }();
  return fn;
}

// [rows, heads, 128] bf16 in boxes of 64 dims x box_heads heads x box_rows rows, 128B swizzle
bool encode_heads(CUtensorMap *m, const void *base, int heads, int rows, int box_heads, int box_rows) {
  auto fn = dec_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {256, (cuuint64_t)heads * 256};
  cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool decode_few_rows_supported(const KernelArgs &a, int kv_rows) {
  auto al = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!dec_encoder()) return false;
  if (!al(a.q) || !al(a.k) || !al(a.v) || !al(a.out)) return false;
  if (a.group <= 0 || a.max_q <= 0 || (long)a.group * a.max_q > NR) return false;   // one item, every row
  if (a.max_q > a.total_q) return false;   // the q box (max_q tokens) fits the tensor
  if (a.rd > 64) return false;             // the R pre-pass holds r rows of 64 at most
  return kv_rows >= KT;                    // K / V boxes of 128 rows
}

bool decode_mxfp8_supported(const KernelArgs &a, const void *k8, const void *v8, const void *ks,
                            const void *vs, int kv_rows) {
  auto al = [](const void *p, uintptr_t n) { return p && (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; };
  if (!dec_encoder()) return false;
  if (!al(a.q, 16) || !al(a.out, 16) || !al(k8, 16) || !al(v8, 16) || !al(ks, 4) || !al(vs, 4)) return false;
  if (a.group <= 0 || a.max_q <= 0 || (long)a.group * a.max_q > NR) return false;
  if (a.rd > 64 || a.block_table != nullptr) return false;
  return kv_rows >= KT;
}

// In-kernel R (bf16 few-row kernel): r rows by TMA (16-byte rows and base),
// r_dim <= 64, and P^T plus one item's R beside S and O in 512 TMEM columns
bool decode_rel_in_kernel(const KernelArgs &a) {
  if (!(a.rd > 0 && a.E > 0) || a.sms <= 0) return false;
  if (a.rd % 8 != 0 || a.rd > 64 || (reinterpret_cast<uintptr_t>(a.r) & 15u) != 0) return false;
  // P [r_dim][E] by TMA: 16-byte rows and base; all of it staged in the V ring at once
  if (a.E % 8 != 0 || (reinterpret_cast<uintptr_t>(a.P) & 15u) != 0) return false;
  const long nt = (a.E + 127) / 128;
  static_assert(kRelMaxBlocks * 128 * 64 * 2 <= Lay<false>::VST * Lay<false>::KTILE, "P fits the V ring");
  return nt <= kRelMaxBlocks && (long)TM_PT + nt * 48 <= kRelTmemCols;
}

int decode_rel_rs(const KernelArgs &a) { return (a.group * a.max_q + 3) / 4 * 4; }

// workspace for either source of R: the rows of every decode row (R kernel,
// MXFP8 decode or a shape the in-kernel path does not take), or two slots per
// CTA (in-kernel)
size_t decode_rel_bytes(const KernelArgs &a) {
  if (!(a.rd > 0 && a.E > 0)) return 0;
  size_t b = (size_t)a.total_q * a.Hq * a.E * sizeof(float);
  if (decode_rel_in_kernel(a)) {
    const size_t slots = (size_t)a.sms * 2 * ((a.E + 127) / 128) * 128 * decode_rel_rs(a) * sizeof(float);
    b = std::max(b, slots);
  }
  return b;
}

cudaError_t launch_decode_few_rows(const KernelArgs &a, int kv_rows, cudaStream_t stream) {
  DecArgs da;
  da.a = a;
  da.kscale = da.vscale = nullptr;
  da.kv_rows = kv_rows;
  da.has_bias = a.rd > 0 && a.E > 0 && a.rdec != nullptr;
  da.q_bytes = 2 * 64 * 2 * a.group * a.max_q;
  const long items = (long)a.num_splits * a.batch * a.Hkv;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffL) return cudaErrorInvalidValue;
  da.n_items = (int)items;
  set_walk(a, da);
  CUtensorMap mq, mk, mv, mr;
  if (!encode_heads(&mq, a.q, a.Hq, a.total_q, a.group, a.max_q) ||
      !encode_heads(&mk, a.k, a.Hkv, kv_rows, 1, KT) || !encode_heads(&mv, a.v, a.Hkv, kv_rows, 1, KT))
    return cudaErrorInvalidValue;
  CUtensorMap mp = mq;
  mr = mq;   // (unused unless R is computed in the kernel)
  da.rel_mode = !da.has_bias ? 0 : decode_rel_in_kernel(a) ? 2 : 1;
  da.nt_e = (a.E + 127) / 128;
  da.rs = decode_rel_rs(a);
  da.r_bytes = 128 * a.group * a.max_q;
  da.rslot = const_cast<float *>(a.rdec);
  if (da.rel_mode == 2) {
    // r [total_q, Hq, r_dim] in boxes of 64 channels x group heads x max_q
    // tokens (channels past r_dim read as 0), 128-byte swizzle
    auto fn = dec_encoder();
    cuuint64_t dims[3] = {(cuuint64_t)a.rd, (cuuint64_t)a.Hq, (cuuint64_t)a.total_q};
    cuuint64_t strides[2] = {(cuuint64_t)a.rd * 2, (cuuint64_t)a.Hq * a.rd * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)a.group, (cuuint32_t)a.max_q};
    cuuint32_t es[3] = {1, 1, 1};
    // P [r_dim, E] in boxes of 128 distances x r_dim channels (distances past
    // E read as 0), no swizzle: [r_dim][128] bf16 per box
    cuuint64_t pdims[2] = {(cuuint64_t)a.E, (cuuint64_t)a.rd};
    cuuint64_t pstrides[1] = {(cuuint64_t)a.E * 2};
    cuuint32_t pbox[2] = {(cuuint32_t)KT, (cuuint32_t)a.rd};
    if (fn(&mr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16 *>(a.r), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        fn(&mp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(a.P), pdims, pstrides, pbox, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      da.rel_mode = 1;
  }
  if (da.rel_mode == 1) {
    // R for the decode rows first (same stream)
    cudaError_t e = launch_decode_rel(a, stream);
    if (e != cudaSuccess) return e;
  }
  static std::atomic<bool> attr_set[kMaxDevicesAttr];
  constexpr uint32_t smem = Lay<false>::SMEM_BYTES;
  cudaError_t e = set_max_smem_once(reinterpret_cast<const void *>(relattn_decode_tc_kernel<false>),
                                    (int)smem, attr_set);
  if (e != cudaSuccess) return e;
  return launch_decode_kernel(relattn_decode_tc_kernel<false>, walk_grid(a, da, items), smem, stream, da, mq,
                              mk, mv, mr, mp, da.rel_mode == 1);
}

cudaError_t launch_decode_mxfp8(const KernelArgs &a, const void *k8, const void *v8, const void *ks,
                                const void *vs, int kv_rows, cudaStream_t stream) {
  DecArgs da;
  da.a = a;
  da.kscale = static_cast<const uint32_t *>(ks);
  da.vscale = static_cast<const uint32_t *>(vs);
  da.kv_rows = kv_rows;
  da.has_bias = a.rd > 0 && a.E > 0 && a.rdec != nullptr;
  da.q_bytes = 0;
  const long items = (long)a.num_splits * a.batch * a.Hkv;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffL) return cudaErrorInvalidValue;
  da.n_items = (int)items;
  set_walk(a, da);
  da.rel_mode = da.has_bias ? 1 : 0;
  da.nt_e = da.rs = da.r_bytes = 0;
  da.rslot = nullptr;
  if (da.has_bias) {
    cudaError_t e = launch_decode_rel(a, stream);
    if (e != cudaSuccess) return e;
  }
  // E4M3 codes [rows, heads, 128] in boxes of 128 dims x 1 head x 128 rows
  auto encode_codes = [](CUtensorMap *m, const void *base, int heads, int rows) {
    auto fn = dec_encoder();
    if (!fn) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {128, (cuuint64_t)heads * 128};
    cuuint32_t box[3] = {128, 1, (cuuint32_t)KT};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  CUtensorMap mk, mv;
  if (!encode_codes(&mk, k8, a.Hkv, kv_rows) || !encode_codes(&mv, v8, a.Hkv, kv_rows))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[kMaxDevicesAttr];
  constexpr uint32_t smem = Lay<true>::SMEM_BYTES;
  cudaError_t e = set_max_smem_once(reinterpret_cast<const void *>(relattn_decode_tc_kernel<true>),
                                    (int)smem, attr_set);
  if (e != cudaSuccess) return e;
  // (the q and r maps are not read: the producer quantises q rows itself,
  // and R comes from the R kernel)
  return launch_decode_kernel(relattn_decode_tc_kernel<true>, walk_grid(a, da, items), smem, stream, da, mk,
                              mk, mv, mk, mk, da.rel_mode == 1);
}

}  // namespace relattn
