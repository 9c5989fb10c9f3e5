// api.cu -- the C ABI (include/relattn.h): argument checks, split planning,
// kernel dispatch.  No allocation, no synchronisation (except the explicit
// relattn_get_device_error), no host fallback.
#include <math.h>

#include <atomic>
#include <mutex>

#include "launch.h"

using namespace relattn;

namespace {

__device__ int g_device_error;

#ifdef RELATTN_TEST_HOOKS
// Test build only (librelattn_test.so): settings the relattn_test_* entry
// points change, read by the launches of the same process.
std::atomic<int> g_test_skip_k_tile{-1};     // K tile the tcgen05 producers never load
std::atomic<int> g_test_band_ctas{0};        // CTA cap of the persistent band / walking launches
std::atomic<int> g_test_prologue_skip{-1};   // token tile whose prologue copies are never issued
std::atomic<int> g_test_bwd_dkdv_skip{-1};   // step the tcgen05 dk / dv producer never loads
std::atomic<int> g_test_bwd_dq_skip{-1};     // step the tcgen05 dq producer never loads
#else
// The product library has no test hooks: these are constants (every hook off).
constexpr int g_test_skip_k_tile = -1;
constexpr int g_test_band_ctas = 0;
constexpr int g_test_prologue_skip = -1;
constexpr int g_test_bwd_dkdv_skip = -1;
constexpr int g_test_bwd_dq_skip = -1;
#endif

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_err_ptr[kMaxDevices];
void *g_err_ctx[kMaxDevices];   // the context g_err_ptr[dev] was looked up in
int g_sms[kMaxDevices];
int g_last_error_word = 0;

relattn_status device_state(int *dev_out, int **err_out, int *sms_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RELATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  void *ctx = current_cu_context();
  if (!g_err_ptr[dev] || !ctx || ctx != g_err_ctx[dev]) {
    // first call on this device, or a new context (after cudaDeviceReset):
    // the error word's address is looked up again in the current one
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return RELATTN_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return RELATTN_ERR_CUDA;
    g_err_ptr[dev] = static_cast<int *>(p);
    g_err_ctx[dev] = current_cu_context();
    g_sms[dev] = sms;
  }
  if (dev_out) *dev_out = dev;
  if (err_out) *err_out = g_err_ptr[dev];
  if (sms_out) *sms_out = g_sms[dev];
  return RELATTN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxRDim = 64;
constexpr int kMaxDecodeRows = 16;

relattn_status validate(const relattn_params *p, bool decode) {
  if (!p) return RELATTN_ERR_INVALID_ARG;
  if (p->head_dim != kHeadDim) return RELATTN_ERR_UNSUPPORTED;
  if (p->num_heads_q <= 0 || p->num_heads_kv <= 0 || p->num_heads_q % p->num_heads_kv != 0)
    return RELATTN_ERR_INVALID_ARG;
  if (p->batch < 0 || p->total_q < 0 || p->total_k < 0 || p->max_seqlen_q < 0 ||
      p->max_seqlen_k < 0 || p->rel_extent < 0 || p->r_dim < 0)
    return RELATTN_ERR_INVALID_ARG;
  if (p->r_dim > kMaxRDim) return RELATTN_ERR_UNSUPPORTED;
  if (!isfinite(p->alpha)) return RELATTN_ERR_INVALID_ARG;
  if (!(p->log_scale_base <= 0.f || (p->log_scale_base > 1.f && isfinite(p->log_scale_base))))
    return RELATTN_ERR_INVALID_ARG;
  if (decode && p->max_seqlen_q > kMaxDecodeRows) return RELATTN_ERR_UNSUPPORTED;
  if (p->batch == 0 || p->total_q == 0) return RELATTN_OK;
  if (p->max_seqlen_q <= 0 || p->max_seqlen_k < p->max_seqlen_q) return RELATTN_ERR_INVALID_ARG;
  if (!p->q || !p->k || !p->v || !p->out || !p->lse || !p->cu_seqlens_q || !p->cu_seqlens_k)
    return RELATTN_ERR_INVALID_ARG;
  if (!aligned16(p->q) || !aligned16(p->k) || !aligned16(p->v) || !aligned16(p->out))
    return RELATTN_ERR_INVALID_ARG;
  if (p->r_dim > 0 && p->rel_extent > 0 && (!p->r || !p->P)) return RELATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(p->lse) & 3u) != 0) return RELATTN_ERR_INVALID_ARG;
  return RELATTN_OK;
}

relattn_status make_args(const relattn_params *p, KernelArgs *a) {
  int *err = nullptr, sms = 0;
  relattn_status st = device_state(nullptr, &err, &sms);
  if (st != RELATTN_OK) return st;
  KernelArgs &x = *a;
  x = KernelArgs{};
  x.q = static_cast<const __nv_bfloat16 *>(p->q);
  x.k = static_cast<const __nv_bfloat16 *>(p->k);
  x.v = static_cast<const __nv_bfloat16 *>(p->v);
  x.r = static_cast<const __nv_bfloat16 *>(p->r);
  x.P = static_cast<const __nv_bfloat16 *>(p->P);
  x.cu_q = p->cu_seqlens_q;
  x.cu_k = p->cu_seqlens_k;
  x.out = static_cast<__nv_bfloat16 *>(p->out);
  x.lse = p->lse;
  x.err = err;
  x.batch = p->batch;
  x.total_q = p->total_q;
  x.max_q = p->max_seqlen_q;
  x.max_k = p->max_seqlen_k;
  x.Hq = p->num_heads_q;
  x.Hkv = p->num_heads_kv;
  x.group = p->num_heads_q / p->num_heads_kv;
  const bool bias = p->r_dim > 0 && p->rel_extent > 0;
  x.rd = bias ? p->r_dim : 0;
  x.rd_pad = bias ? (p->r_dim + 15) / 16 * 16 : 0;
  x.E = bias ? p->rel_extent : 0;
  x.window = p->window > 0 ? p->window : 0;
  x.alpha_log2e = p->alpha * kLog2e;
  x.inv_ln_base = p->log_scale_base > 1.f ? 1.f / logf(p->log_scale_base) : 0.f;
  x.r_vec_ok = bias && (p->r_dim % 8 == 0) && aligned16(p->r);
  x.test_skip_k_tile = g_test_skip_k_tile;
  x.p_vec_ok = bias && (p->rel_extent % 8 == 0) && aligned16(p->P);
  x.num_splits = 1;
  x.split_chunk = 0;
  x.q_tiles = (p->max_seqlen_q + 127) / 128;
  x.row_blocks = 1;
  const int band_ctas = g_test_band_ctas;
  x.sms = band_ctas > 0 ? band_ctas : sms;
  return RELATTN_OK;
}

// Decode kernels: few rows per (sequence, kv head) -- the keys along the
// MMA's M (decode_tc.cu) --, else 128-row blocks on the prefill kernel
// (fwd_tc.cu), else the warp-MMA kernel (fwd_mma.cu) where the tcgen05
// kernels' alignment or shape conditions fail.
enum class DecodeKind { kMma, kRows, kKeys };

struct DecodePlan {
  DecodeKind kind;
  int warps, row_blocks, splits, chunk;
  // workspace: split partials (o, then lse at lse_offset) when splits > 1,
  // then (few-row kernel with a bias) R of the decode rows at rel_offset
  size_t ws_bytes, lse_offset, rel_offset;
  bool tc() const { return kind != DecodeKind::kMma; }
};

// kv_rows: rows of the K / V tensors the kernels address (total_k, or the
// page pool's rows for paged K / V)
relattn_status plan_decode(const relattn_params *p, DecodePlan *plan, long kv_rows = -1) {
  int sms = 0;
  relattn_status st = device_state(nullptr, nullptr, &sms);
  if (st != RELATTN_OK) return st;
  const int group = p->num_heads_q / p->num_heads_kv;
  const int rows = p->max_seqlen_q * group;
  KernelArgs probe;
  if ((st = make_args(p, &probe)) != RELATTN_OK) return st;
  const int kvr = kv_rows >= 0 ? (int)kv_rows : p->total_k;
  plan->kind = decode_few_rows_supported(probe, kvr) ? DecodeKind::kKeys
               : tc_supported(probe, kvr)            ? DecodeKind::kRows
                                                     : DecodeKind::kMma;
  plan->warps = decode_warps_for_rows(rows < 128 ? rows : 128);
  const int m = plan->kind == DecodeKind::kKeys   ? kFewRows
                : plan->kind == DecodeKind::kRows ? kTcDecodeRows
                                                  : plan->warps * 16;
  plan->row_blocks = (rows + m - 1) / m;
  const int tile = plan->tc() ? kTcKeyTile : kDecodeKeyTile;
  // keys any CTA of one (sequence, kv head) may visit, from an aligned start
  long max_vis = p->max_seqlen_k;
  if (p->window > 0) {
    const long w = (long)p->window + p->max_seqlen_q - 1 + (tile - 1);
    if (w < max_vis) max_vis = w;
  }
  if (max_vis < 1) max_vis = 1;
  long chunk;
  if (p->num_splits > 0) {
    chunk = (max_vis + p->num_splits - 1) / p->num_splits;
  } else {
    // keys all CTAs visit together (each sequence sees at most max_vis of its
    // keys), cut into one wave of CTAs when there are few (sequence, kv head,
    // row block) units -- long sequences split evenly, one CTA per SM -- and
    // into about two waves otherwise, where splits past a short sequence's
    // keys exit at once and the second wave evens out variable lengths
    long seq_keys = (long)p->total_k;
    if ((long)p->batch * max_vis < seq_keys) seq_keys = (long)p->batch * max_vis;
    const long units = (long)p->batch * p->num_heads_kv * plan->row_blocks;
    const long work = seq_keys * p->num_heads_kv * plan->row_blocks;
    const long target = (2 * units <= sms ? 1L : 2L) * sms;
    chunk = (work + target - 1) / target;
    if (chunk < 256) chunk = 256;                       // at least 256 keys per split
    // sliding window on the few-row kernel: when every sequence holds a full
    // window (all units the same size) and the units about fill the SMs, one
    // split each -- a CTA then runs at most one item, and no item boundary
    // (each costs the length of a few tiles in that kernel) or combine is paid
    if (plan->kind == DecodeKind::kKeys && p->window > 0 && seq_keys == (long)p->batch * max_vis &&
        4 * units >= 3L * sms && units <= sms)
      chunk = max_vis;
  }
  chunk = (chunk + tile - 1) / tile * tile;
  if (chunk > (max_vis + tile - 1) / tile * tile) chunk = (max_vis + tile - 1) / tile * tile;
  long splits = (max_vis + chunk - 1) / chunk;
  if (splits > 65535) return RELATTN_ERR_UNSUPPORTED;
  plan->splits = (int)splits;
  plan->chunk = (int)chunk;
  size_t end = 0;
  plan->lse_offset = 0;
  if (plan->splits > 1) {
    const size_t rows_all = (size_t)p->total_q * p->num_heads_q;
    const size_t o_bytes = (size_t)plan->splits * rows_all * kHeadDim * sizeof(float);
    plan->lse_offset = (o_bytes + 255) / 256 * 256;
    end = plan->lse_offset + (size_t)plan->splits * rows_all * sizeof(float);
  }
  plan->rel_offset = (end + 255) / 256 * 256;
  const size_t rel = plan->kind == DecodeKind::kKeys ? decode_rel_bytes(probe) : 0;
  plan->ws_bytes = rel > 0 ? plan->rel_offset + rel : end;
  return RELATTN_OK;
}

relattn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? RELATTN_OK : RELATTN_ERR_CUDA; }

bool aligned(const void *p, uintptr_t bytes) {
  return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) == 0;
}

// [a, a + na) and [b, b + nb) share a byte
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

// D [Hq, Tq], then (with a bias) R = r . P [Tq, Hq, E rounded up to 4] and
// the partial dq [Tq, Hq, 128], both fp32
size_t backward_d_bytes(const relattn_params &f) {
  return ((size_t)f.num_heads_q * f.total_q * sizeof(float) + 255) / 256 * 256;
}
size_t backward_rall_bytes(const relattn_params &f) {
  if (!(f.r_dim > 0 && f.rel_extent > 0)) return 0;
  return (size_t)f.total_q * f.num_heads_q * ((f.rel_extent + 3) / 4 * 4) * sizeof(float);
}
size_t backward_dq_part_bytes(const relattn_params &f) {
  if (!(f.r_dim > 0 && f.rel_extent > 0)) return 0;
  return (size_t)f.total_q * f.num_heads_q * kHeadDim * sizeof(float);
}
// two fp32 halves of dk and dv when the GQA group is even and at least 4 (the
// tcgen05 dk / dv then splits a group's query heads between two CTAs)
size_t backward_dkv_part_bytes(const relattn_params &f) {
  const int group = f.num_heads_kv > 0 ? f.num_heads_q / f.num_heads_kv : 0;
  if (group < 4 || group % 2) return 0;
  return (size_t)4 * f.total_k * f.num_heads_kv * kHeadDim * sizeof(float);
}
size_t backward_workspace_bytes(const relattn_params &f) {
  return backward_d_bytes(f) + backward_rall_bytes(f) + backward_dq_part_bytes(f) + backward_dkv_part_bytes(f);
}

relattn_status validate_backward(const relattn_bwd_params *p) {
  if (!p) return RELATTN_ERR_INVALID_ARG;
  const relattn_params &f = p->fwd;
  relattn_status st = validate(&f, false);
  if (st != RELATTN_OK) return st;
  if (f.r_dim % 8 != 0) return RELATTN_ERR_UNSUPPORTED;
  if (f.batch == 0) return RELATTN_OK;
  if (f.total_k > 0 && (!p->dk || !p->dv || !aligned16(p->dk) || !aligned16(p->dv)))
    return RELATTN_ERR_INVALID_ARG;
  if (f.total_q == 0) return RELATTN_OK;
  if (!p->dout || !p->dq || !aligned16(p->dout) || !aligned16(p->dq) || !aligned16(f.lse))
    return RELATTN_ERR_INVALID_ARG;
  if (f.r_dim > 0 && (!p->dr || !aligned16(p->dr))) return RELATTN_ERR_INVALID_ARG;
  if (f.r_dim > 0 && f.rel_extent > 0 && (!aligned16(f.r) || !aligned16(f.P)))
    return RELATTN_ERR_INVALID_ARG;
  if (!p->workspace || !aligned16(p->workspace) || p->workspace_bytes < backward_workspace_bytes(f))
    return RELATTN_ERR_WORKSPACE;
  return RELATTN_OK;
}

relattn_status validate_prologue(const relattn_prologue_params *p, const relattn_kv_mxfp8_out *mx = nullptr) {
  if (!p) return RELATTN_ERR_INVALID_ARG;
  if (p->head_dim != kHeadDim) return RELATTN_ERR_UNSUPPORTED;
  if (p->batch < 0 || p->total_q < 0 || p->total_k < 0 || p->num_heads_q <= 0 ||
      p->num_heads_kv <= 0 || p->num_heads_q % p->num_heads_kv != 0)
    return RELATTN_ERR_INVALID_ARG;
  if (!(isfinite(p->eps) && p->eps > 0.f)) return RELATTN_ERR_INVALID_ARG;
  if (p->batch == 0) return RELATTN_OK;
  const void *need[] = {p->q, p->k, p->v, p->q_out, p->conv_k, p->conv_v, p->norm_q, p->norm_k};
  for (const void *x : need)
    if (!x || !aligned(x, 16)) return RELATTN_ERR_INVALID_ARG;
  // the bf16 cache is optional only when an MXFP8 one is written
  const void *caches[] = {p->k_cache, p->v_cache};
  for (const void *x : caches)
    if (mx ? (x && !aligned(x, 16)) : (!x || !aligned(x, 16))) return RELATTN_ERR_INVALID_ARG;
  if (mx) {
    if (!mx->k || !mx->v || !mx->k_scale || !mx->v_scale || !aligned(mx->k, 8) || !aligned(mx->v, 8))
      return RELATTN_ERR_INVALID_ARG;
    const size_t codes = (size_t)p->total_k * p->num_heads_kv * kHeadDim, sc = codes / 32;
    const size_t in_bytes = (size_t)p->total_q * p->num_heads_kv * kHeadDim * 2;
    const void *outs8[] = {mx->k, mx->v, mx->k_scale, mx->v_scale};
    const size_t n8[] = {codes, codes, sc, sc};
    for (int i = 0; i < 4; ++i)
      if (overlaps(outs8[i], n8[i], p->k, in_bytes) || overlaps(outs8[i], n8[i], p->v, in_bytes))
        return RELATTN_ERR_INVALID_ARG;
  }
  if (!p->cu_seqlens_q || !p->cu_seqlens_k) return RELATTN_ERR_INVALID_ARG;
  const void *states[] = {p->conv_state_in_k, p->conv_state_in_v, p->conv_state_out_k,
                          p->conv_state_out_v};
  for (const void *x : states)
    if (x && !aligned(x, 16)) return RELATTN_ERR_INVALID_ARG;
  const size_t row = (size_t)kHeadDim * 2;
  const size_t q_bytes = (size_t)p->total_q * p->num_heads_q * row;
  const size_t kv_bytes = (size_t)p->total_q * p->num_heads_kv * row;
  const size_t cache_bytes = (size_t)p->total_k * p->num_heads_kv * row;
  const size_t state_bytes = (size_t)p->batch * 3 * p->num_heads_kv * row;
  if (p->q_out != p->q && overlaps(p->q_out, q_bytes, p->q, q_bytes)) return RELATTN_ERR_INVALID_ARG;
  const void *kv_in[] = {p->k, p->v};
  for (const void *x : kv_in)
    if (overlaps(p->k_cache, cache_bytes, x, kv_bytes) || overlaps(p->v_cache, cache_bytes, x, kv_bytes))
      return RELATTN_ERR_INVALID_ARG;
  const void *outs[] = {p->conv_state_out_k, p->conv_state_out_v};
  for (const void *o : outs)
    if (o && (overlaps(o, state_bytes, p->conv_state_in_k, p->conv_state_in_k ? state_bytes : 0) ||
              overlaps(o, state_bytes, p->conv_state_in_v, p->conv_state_in_v ? state_bytes : 0)))
      return RELATTN_ERR_INVALID_ARG;
  return RELATTN_OK;
}

}  // namespace

extern "C" {

relattn_status relattn_prefill(const relattn_params *p, void *stream) {
  relattn_status st = validate(p, false);
  if (st != RELATTN_OK) return st;
  if (p->batch == 0 || p->total_q == 0) return RELATTN_OK;
  KernelArgs a;
  if ((st = make_args(p, &a)) != RELATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (tc_supported(a, p->total_k)) {
    if (tc_main_supported(a, p->total_q, p->total_k)) {
      // the bias band on the bias kernel (out / lse normalised over the band),
      // then every other key tile on the two-head main kernel, which starts
      // from that state
      if (a.rd > 0 && a.E > 0) {
        a.band_only = 1;
        cudaError_t e = launch_prefill_tc(a, p->total_k, s);
        if (e != cudaSuccess) return cuda_status(e);
        a.band_only = 0;
        a.init_from_out = 1;
      }
      return cuda_status(launch_prefill_tc_main(a, p->total_k, s));
    }
    return cuda_status(launch_prefill_tc(a, p->total_k, s));
  }
  return cuda_status(launch_prefill_mma(a, s));
}

relattn_status relattn_decode_workspace_size(const relattn_params *p, size_t *bytes) {
  if (!bytes) return RELATTN_ERR_INVALID_ARG;
  relattn_status st = validate(p, true);
  if (st != RELATTN_OK) return st;
  *bytes = 0;
  if (p->batch == 0 || p->total_q == 0) return RELATTN_OK;
  DecodePlan plan;
  if ((st = plan_decode(p, &plan)) != RELATTN_OK) return st;
  *bytes = plan.ws_bytes;
  return RELATTN_OK;
}

relattn_status relattn_decode_num_splits(const relattn_params *p, int32_t *num_splits) {
  if (!num_splits) return RELATTN_ERR_INVALID_ARG;
  relattn_status st = validate(p, true);
  if (st != RELATTN_OK) return st;
  *num_splits = 1;
  if (p->batch == 0 || p->total_q == 0) return RELATTN_OK;
  DecodePlan plan;
  if ((st = plan_decode(p, &plan)) != RELATTN_OK) return st;
  *num_splits = plan.splits;
  return RELATTN_OK;
}

// the split kernel, then the combine when there are several splits; kv_rows:
// rows the K / V tensors hold
relattn_status run_decode(const relattn_params *p, const DecodePlan &plan, KernelArgs &a, long kv_rows,
                          cudaStream_t s, const relattn_kv_mxfp8 *f8 = nullptr) {
  a.num_splits = plan.splits;
  a.split_chunk = plan.chunk;
  a.row_blocks = plan.row_blocks;
  if (plan.ws_bytes > 0) {
    if (!p->workspace || p->workspace_bytes < plan.ws_bytes || !aligned16(p->workspace))
      return RELATTN_ERR_WORKSPACE;
    char *ws = static_cast<char *>(p->workspace);
    if (plan.splits > 1) {
      a.o_part = reinterpret_cast<float *>(ws);
      a.lse_part = reinterpret_cast<float *>(ws + plan.lse_offset);
    }
    if (plan.kind == DecodeKind::kKeys && decode_rel_bytes(a) > 0)
      a.rdec = reinterpret_cast<const float *>(ws + plan.rel_offset);
  }
  cudaError_t e;
  switch (plan.kind) {
    case DecodeKind::kKeys:
      e = f8 ? launch_decode_mxfp8(a, f8->k, f8->v, f8->k_scale, f8->v_scale, (int)kv_rows, s)
             : launch_decode_few_rows(a, (int)kv_rows, s);
      break;
    case DecodeKind::kRows: e = launch_decode_tc(a, (int)kv_rows, s); break;
    default: e = launch_decode_mma(a, plan.warps, s); break;
  }
  relattn_status st = cuda_status(e);
  if (st != RELATTN_OK) return st;
  if (plan.splits > 1)
    st = cuda_status(launch_combine(a.o_part, a.lse_part, plan.splits, p->total_q,
                                    p->num_heads_q, a.out, a.lse, s, plan.kind == DecodeKind::kKeys));
  return st;
}

relattn_status relattn_decode(const relattn_params *p, void *stream) {
  relattn_status st = validate(p, true);
  if (st != RELATTN_OK) return st;
  if (p->batch == 0 || p->total_q == 0) return RELATTN_OK;
  DecodePlan plan;
  if ((st = plan_decode(p, &plan)) != RELATTN_OK) return st;
  KernelArgs a;
  if ((st = make_args(p, &a)) != RELATTN_OK) return st;
  return run_decode(p, plan, a, p->total_k, static_cast<cudaStream_t>(stream));
}

relattn_status relattn_decode_paged(const relattn_params *p, const relattn_paged_kv *kv,
                                   void *stream) {
  relattn_status st = validate(p, true);
  if (st != RELATTN_OK) return st;
  if (!kv) return RELATTN_ERR_INVALID_ARG;
  if (kv->page_size <= 0 || kv->page_size % kTcKeyTile != 0) return RELATTN_ERR_UNSUPPORTED;
  if (kv->num_pages <= 0 || kv->max_pages_per_seq <= 0) return RELATTN_ERR_INVALID_ARG;
  if ((long)kv->num_pages * kv->page_size > 0x7fffffffL) return RELATTN_ERR_UNSUPPORTED;
  if ((long)kv->max_pages_per_seq * kv->page_size < p->max_seqlen_k) return RELATTN_ERR_INVALID_ARG;
  if (!kv->block_table || (reinterpret_cast<uintptr_t>(kv->block_table) & 3u) != 0)
    return RELATTN_ERR_INVALID_ARG;
  if (p->batch == 0 || p->total_q == 0) return RELATTN_OK;
  const long pool_rows = (long)kv->num_pages * kv->page_size;
  DecodePlan plan;
  if ((st = plan_decode(p, &plan, pool_rows)) != RELATTN_OK) return st;
  if (!plan.tc()) return RELATTN_ERR_UNSUPPORTED;   // paged K / V: the tcgen05 kernels only
  KernelArgs a;
  if ((st = make_args(p, &a)) != RELATTN_OK) return st;
  a.block_table = kv->block_table;
  a.page_size = kv->page_size;
  a.max_pages = kv->max_pages_per_seq;
  a.num_pages = kv->num_pages;
  return run_decode(p, plan, a, pool_rows, static_cast<cudaStream_t>(stream));
}

relattn_status relattn_decode_mxfp8(const relattn_params *p, const relattn_kv_mxfp8 *kv, void *stream) {
  if (!p || !kv) return RELATTN_ERR_INVALID_ARG;
  // the code tensors stand in for k / v in the checks and the plan
  relattn_params q = *p;
  q.k = kv->k;
  q.v = kv->v;
  relattn_status st = validate(&q, true);
  if (st != RELATTN_OK) return st;
  if (q.batch == 0 || q.total_q == 0) return RELATTN_OK;
  if (!kv->k_scale || !kv->v_scale) return RELATTN_ERR_INVALID_ARG;
  DecodePlan plan;
  if ((st = plan_decode(&q, &plan)) != RELATTN_OK) return st;
  KernelArgs a;
  if ((st = make_args(&q, &a)) != RELATTN_OK) return st;
  if (plan.kind != DecodeKind::kKeys ||
      !decode_mxfp8_supported(a, kv->k, kv->v, kv->k_scale, kv->v_scale, q.total_k))
    return RELATTN_ERR_UNSUPPORTED;
  return run_decode(&q, plan, a, q.total_k, static_cast<cudaStream_t>(stream), kv);
}

relattn_status relattn_quantize_mxfp8(const void *x, int64_t n_blocks, void *codes, void *scales,
                                      void *stream) {
  if (n_blocks < 0) return RELATTN_ERR_INVALID_ARG;
  if (n_blocks == 0) return RELATTN_OK;
  if (!x || !codes || !scales || !aligned16(x) || !aligned16(codes)) return RELATTN_ERR_INVALID_ARG;
  if (overlaps(x, (size_t)n_blocks * 64, codes, (size_t)n_blocks * 32) ||
      overlaps(x, (size_t)n_blocks * 64, scales, (size_t)n_blocks))
    return RELATTN_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_mxfp8(x, n_blocks, codes, scales, static_cast<cudaStream_t>(stream)));
}

relattn_status relattn_combine(const float *o_part, const float *lse_part, int32_t num_splits,
                               int32_t total_q, int32_t num_heads, void *out, float *lse,
                               void *stream) {
  if (num_splits <= 0 || total_q < 0 || num_heads <= 0) return RELATTN_ERR_INVALID_ARG;
  if (total_q == 0) return RELATTN_OK;
  if (!o_part || !lse_part || !out || !lse || !aligned16(o_part) || !aligned16(out))
    return RELATTN_ERR_INVALID_ARG;
  return cuda_status(launch_combine(o_part, lse_part, num_splits, total_q, num_heads,
                                    static_cast<__nv_bfloat16 *>(out), lse,
                                    static_cast<cudaStream_t>(stream)));
}

relattn_status relattn_backward_workspace_size(const relattn_bwd_params *p, size_t *bytes) {
  if (!bytes || !p) return RELATTN_ERR_INVALID_ARG;
  relattn_status st = validate(&p->fwd, false);
  if (st != RELATTN_OK) return st;
  *bytes = backward_workspace_bytes(p->fwd);
  return RELATTN_OK;
}

relattn_status relattn_backward(const relattn_bwd_params *p, void *stream) {
  relattn_status st = validate_backward(p);
  if (st != RELATTN_OK) return st;
  const relattn_params &f = p->fwd;
  if (f.batch == 0) return RELATTN_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (f.total_q == 0) {   // no query sees any key: the key gradients are zero
    const size_t n = (size_t)f.total_k * f.num_heads_kv * kHeadDim * 2;
    if (n == 0) return RELATTN_OK;
    if (cudaMemsetAsync(p->dk, 0, n, s) != cudaSuccess) return RELATTN_ERR_CUDA;
    return cudaMemsetAsync(p->dv, 0, n, s) == cudaSuccess ? RELATTN_OK : RELATTN_ERR_CUDA;
  }
  int *err = nullptr, sms = 0;
  if ((st = device_state(nullptr, &err, &sms)) != RELATTN_OK) return st;
  BwdArgs a{};
  a.q = static_cast<const __nv_bfloat16 *>(f.q);
  a.k = static_cast<const __nv_bfloat16 *>(f.k);
  a.v = static_cast<const __nv_bfloat16 *>(f.v);
  a.r = static_cast<const __nv_bfloat16 *>(f.r);
  a.P = static_cast<const __nv_bfloat16 *>(f.P);
  a.out = static_cast<const __nv_bfloat16 *>(f.out);
  a.dout = static_cast<const __nv_bfloat16 *>(p->dout);
  a.lse = f.lse;
  a.cu_q = f.cu_seqlens_q;
  a.cu_k = f.cu_seqlens_k;
  a.dq = static_cast<__nv_bfloat16 *>(p->dq);
  a.dk = static_cast<__nv_bfloat16 *>(p->dk);
  a.dv = static_cast<__nv_bfloat16 *>(p->dv);
  a.dr = f.r_dim > 0 ? static_cast<__nv_bfloat16 *>(p->dr) : nullptr;
  a.Dsum = static_cast<float *>(p->workspace);
  a.Rall = reinterpret_cast<float *>(static_cast<char *>(p->workspace) + backward_d_bytes(f));
  a.e_pad = (f.rel_extent + 3) / 4 * 4;
  a.dq_part = reinterpret_cast<float *>(static_cast<char *>(p->workspace) + backward_d_bytes(f) +
                                        backward_rall_bytes(f));
  a.dq_split = 0;              // (set by the launcher)
  a.rall_ok = 0;
  a.dkv_part = backward_dkv_part_bytes(f) ? reinterpret_cast<float *>(
                   static_cast<char *>(p->workspace) + backward_d_bytes(f) + backward_rall_bytes(f) +
                   backward_dq_part_bytes(f)) : nullptr;
  a.kv_split = 1;              // (set by the launcher)
  a.test_skip_dkdv_step = g_test_bwd_dkdv_skip;
  a.test_skip_dq_step = g_test_bwd_dq_skip;
  a.err = err;
  a.batch = f.batch;
  a.total_q = f.total_q;
  a.total_k = f.total_k;
  a.max_q = f.max_seqlen_q;
  a.max_k = f.max_seqlen_k;
  a.Hq = f.num_heads_q;
  a.Hkv = f.num_heads_kv;
  a.group = f.num_heads_q / f.num_heads_kv;
  const bool bias = f.r_dim > 0 && f.rel_extent > 0;
  a.rd = f.r_dim;
  a.rd_pad = bias ? (f.r_dim + 15) / 16 * 16 : 0;
  a.E = bias ? f.rel_extent : 0;
  a.window = f.window > 0 ? f.window : 0;
  a.alpha = f.alpha;
  a.alpha_log2e = f.alpha * kLog2e;
  a.inv_ln_base = f.log_scale_base > 1.f ? 1.f / logf(f.log_scale_base) : 0.f;
  a.p_vec_ok = bias && f.rel_extent % 8 == 0;
  a.q_tiles = (f.max_seqlen_q + 63) / 64;
  a.k_tiles = (f.max_seqlen_k + 63) / 64;
  return cuda_status(launch_backward(a, sms, s));
}

relattn_status relattn_prologue(const relattn_prologue_params *p, void *stream) {
  relattn_status st = validate_prologue(p);
  if (st != RELATTN_OK) return st;
  if (p->batch == 0) return RELATTN_OK;
  int *err = nullptr;
  int sms = 0;
  if ((st = device_state(nullptr, &err, &sms)) != RELATTN_OK) return st;
  return cuda_status(launch_prologue(p, err, sms, g_test_prologue_skip,
                                     static_cast<cudaStream_t>(stream)));
}

relattn_status relattn_prologue_mxfp8(const relattn_prologue_params *p, const relattn_kv_mxfp8_out *cache,
                                      void *stream) {
  if (!cache) return RELATTN_ERR_INVALID_ARG;
  relattn_status st = validate_prologue(p, cache);
  if (st != RELATTN_OK) return st;
  if (p->batch == 0) return RELATTN_OK;
  int *err = nullptr;
  int sms = 0;
  if ((st = device_state(nullptr, &err, &sms)) != RELATTN_OK) return st;
  return cuda_status(launch_prologue(p, err, sms, g_test_prologue_skip,
                                     static_cast<cudaStream_t>(stream), cache));
}

relattn_status relattn_get_device_error(void *stream) {
  int *err = nullptr;
  relattn_status st = device_state(nullptr, &err, nullptr);
  if (st != RELATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host = 0;
  if (cudaMemcpyAsync(&host, err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return RELATTN_ERR_CUDA;
  if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) return RELATTN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RELATTN_ERR_CUDA;
  g_last_error_word = host;
  if (host & kDevErrTimeout) return RELATTN_ERR_TIMEOUT;
  if (host & kDevErrSeqlens) return RELATTN_ERR_DEVICE_ARGS;
  return RELATTN_OK;
}

const char *relattn_status_string(relattn_status s) {
  switch (s) {
    case RELATTN_OK: return "RELATTN_OK";
    case RELATTN_ERR_INVALID_ARG: return "RELATTN_ERR_INVALID_ARG";
    case RELATTN_ERR_UNSUPPORTED: return "RELATTN_ERR_UNSUPPORTED";
    case RELATTN_ERR_CUDA: return "RELATTN_ERR_CUDA";
    case RELATTN_ERR_TIMEOUT: return "RELATTN_ERR_TIMEOUT";
    case RELATTN_ERR_WORKSPACE: return "RELATTN_ERR_WORKSPACE";
    case RELATTN_ERR_DEVICE_ARGS: return "RELATTN_ERR_DEVICE_ARGS";
  }
  return "RELATTN_ERR_UNKNOWN";
}

const char *relattn_version(void) { return "relattn 0.1 sm_103a"; }

int32_t relattn_last_device_error_word(void) { return g_last_error_word; }

#ifdef RELATTN_TEST_HOOKS
relattn_status relattn_test_skip_k_tile(int32_t tile) {
  if (tile < -1) return RELATTN_ERR_INVALID_ARG;
  g_test_skip_k_tile = tile;
  return RELATTN_OK;
}

relattn_status relattn_test_prologue_skip_tile(int32_t tile) {
  if (tile < -1) return RELATTN_ERR_INVALID_ARG;
  g_test_prologue_skip = tile;
  return RELATTN_OK;
}

relattn_status relattn_test_backward_skip_step(int32_t kernel, int32_t step) {
  if (step < -1 || kernel < 0 || kernel > 1) return RELATTN_ERR_INVALID_ARG;
  (kernel == 0 ? g_test_bwd_dkdv_skip : g_test_bwd_dq_skip) = step;
  return RELATTN_OK;
}

relattn_status relattn_test_band_ctas(int32_t n) {
  if (n < 0) return RELATTN_ERR_INVALID_ARG;
  g_test_band_ctas = n;
  return RELATTN_OK;
}
#endif  // RELATTN_TEST_HOOKS

}  // extern "C"
