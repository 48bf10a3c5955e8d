// Host side of the split-KV verify attention for EAGLE target-verify at
// topk = 1, for GB300 (sm_103a): the C ABI of include/verify_splitkv.h, the
// gate, the call plans and the launches.  The operation is defined on the
// sglang "verify_splitkv.py" page (module docstring; "_verify_prefix_stage1",
// "_verify_combine_stage2", "verify_splitkv_fwd", "can_handle"); the kernels
// are in verify_kernel.cuh.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/verify_splitkv.h"
#include "verify_kernel.cuh"
#include "verify_tr.cuh"

#define VSK_VERSION "verify_splitkv-gb300 0.2"

namespace vsk {

// Host-side policy of the planner: which form a call takes and how it is cut
// (prefix tokens x KV heads are from static shapes: kv_indices entries, or
// block-table capacity, times h_kv).
constexpr long long kTwoTileMinTokens = 65536;  // one-launch kernel: prefix tokens from which warps take two tiles
constexpr long long kDefaultMinTokens = 64;  // smallest CTA share of the flattened token space
constexpr long long kPiecesPerSegment = 24;    // ... and at least the mean prefix over this many (one launch)
constexpr long long kPiecesPerSegmentColSplit = 48;  // ... over this many for the two-launch and cluster forms
constexpr long long kColSplitEndBf16 = 1LL << 18;  // head_dim 256: column split below this many token-heads (bf16)
constexpr long long kColSplitEndE4m3 = 1LL << 17;  // ... (e4m3 pools); from there the stream-only kernel + combine
constexpr long long kSplit256MaxWork = 1LL << 23;   // ... up to which head_dim 256 takes the stream-only kernel + combine
// head_dim 256, <= 32 packed rows: the rows-on-M tensor-memory stream + combine
// (measured faster) for e4m3 pools with 17-32 rows, or <= 16 rows below
// kRowsMR16EndE4m3; for bf16 pools with <= 16 rows, or 17-32 rows below
// kRowsMEndBf16; never past kSplit256MaxWork (the one-launch kernel there)
constexpr long long kRowsMR16EndE4m3 = 1LL << 20;
constexpr long long kRowsMEndBf16 = 3LL << 18;
constexpr long long kSplitLaunchMaxWork = 1LL << 22;   // head_dim 64 / 128: stream-only + combine up to (R > 16)
constexpr long long kSplitLaunchMaxWork16 = 1LL << 23;  // ... (at most 16 packed rows)
constexpr long long kSplitTwoTileMinTokens = 1LL << 18;  // prefix tokens from which their warps take two tiles
constexpr long long kPdlMaxWork = 1LL << 16;  // token-heads up to which the combine launch is a programmatic dependent
constexpr long long kClMaxWork = 2047;  // cluster form, mode 1: token-heads up to which calls take it
constexpr long long kClMaxSeg = 512;         // ... with at most this many (sequence, KV head) segments
constexpr long long kClTokensPerCta = 64;    // prefix tokens per CTA the cluster size aims at
constexpr int kClMax = 16;                   // CTAs per cluster at most (8 where 16 do not fit an SM group)
// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
thread_local std::string g_err;

int fail(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return 0;
}

// process-wide tuning overrides (0 = default)
int g_num_ctas = 0;
long long g_min_tokens = 0;
int g_max_stages = 0;
int g_max_heads = 0;
int g_tiles = 0;  // tiles per warp override (0 = default)
int g_tc = 3;     // tensor-memory stream for head_dim 256: 3 rows on M by pool and size (default), 2 / 1 rows / keys on M always, 0 never
int g_cs = 1;     // column-split stream for head_dim 256: 1 below kColSplitEnd*, 2 always, 0 never
int g_sl = 1;     // stream + combine launches for head_dim 64 / 128: 1 below kSplitLaunchMaxWork, 2 always, 0 never
int g_cs2 = 1;    // two-tile column split at head_dim 256: 2 always; 0 and 1 (the default) never
int g_cl = 0;     // cluster form: 0 never (the default), 1 up to kClMaxWork, 2 always (where it applies)
int g_pipe = 1;   // head_dim 256 one-launch kernel over e4m3 pools with pipelined stages (1) or not (0)
int g_pdl = 1;    // combine kernel as a programmatic dependent of the stream: 1 up to kPdlMaxWork, 2 always, 0 never

struct Plan {
  int gq, R, MT, MTW, HC, n_hg, nwc, threads, ek;
  int stage_bytes, nst, ring_off, head_bytes, misc_off, misc_bytes;
  size_t smem;
  int ctas_per_sm;
};

int floor_pow2(int x) {
  int r = 1;
  while (r * 2 <= x) r *= 2;
  return r;
}

// Chooses the CTA shape: HC KV heads per CTA x MT 16-row tiles per head; a
// consumer warp owns MTW tiles (two at head_dim <= 128 when a head has more
// than one tile, so its K / V fragments feed both); ring depth from the
// shared-memory budget.  DV: the value head_dim (0: the same as D).
bool make_plan(long long h_q, long long h_kv, long long D, long long L, bool fp8, Plan& pl,
               long long total_tokens, int tiles, long long DV = 0, int hc_cap = 0) {
  if (DV == 0) DV = D;
  if (h_kv <= 0 || h_q % h_kv != 0) return fail("h_q (%lld) must be a positive multiple of h_kv (%lld)", h_q, h_kv);
  const long long R = (h_q / h_kv) * L;
  const long long DM = std::max(D, DV);
  const int maxw = DM > 128 ? 4 : 8;
  if (R > 16LL * maxw) return fail("packed rows (h_q/h_kv)*l_ext = %lld exceed %d for head_dim %lld", R, 16 * maxw, DM);
  pl.gq = static_cast<int>(h_q / h_kv);
  pl.R = static_cast<int>(R);
  int mt = 1;
  while (16 * mt < R) mt *= 2;
  pl.MT = mt;
  // two tiles per warp pay off once there is enough prefix to stream;
  // small problems are latency bound and want more, lighter warps
  if (tiles == 0) tiles = g_tiles;
  if (tiles == 0) tiles = total_tokens >= kTwoTileMinTokens ? 2 : 1;
  pl.MTW = (DM <= 128 && D == DV && mt >= 2 && tiles == 2) ? 2 : 1;
  const int wph = mt / pl.MTW;  // warps per head
  int hc = 1;
  const int hcc = hc_cap > 0 ? hc_cap : (g_max_heads > 0 ? g_max_heads : maxw);
  while (hc * 2 * wph <= maxw && hc * 2 <= hcc && h_kv % (hc * 2) == 0) hc *= 2;
  pl.HC = hc;
  pl.n_hg = static_cast<int>(h_kv / hc);
  pl.nwc = hc * wph;
  pl.threads = pl.nwc * 32;
  pl.ek = fp8 ? 1 : 2;
  // per head: nst stages of 16 K rows + 16 V rows; per warp: the index ring,
  // the mask ring and (two-tile warps; e4m3 pools at head_dim 256) the query tiles
  pl.stage_bytes = kStageTokens * static_cast<int>(D + DV) * pl.ek;
  const int qsm_tiles = (fp8 && D == 256) ? 1 : (pl.MTW == 2 ? 2 : 0);  // query tiles kept in shared memory
  const int fixed = kIdxRing * 128 + 128 + qsm_tiles * 16 * static_cast<int>(D) * 2;
  // CTAs per SM: as many as keep about 8 warps per SM with a ring of at
  // least 3 stages (2 if nothing better fits)
  const int kmax = pl.nwc >= 8 ? 1 : (pl.nwc >= 4 ? 2 : 4);
  const int cap = g_max_stages > 0 ? std::min(g_max_stages, kMaxStages) : kMaxStages;
  pl.nst = 0;
  for (int want = 3; want >= 2 && pl.nst == 0; --want) {
    for (int k = kmax; k >= 1; --k) {
      const int budget = std::min(kSmemPerCTAMax, kSmemPerSM / k - kReservedPerCTA);
      const int nst = std::min(cap, (budget - kCtlBytes - pl.nwc * fixed) / (pl.HC * pl.stage_bytes));
      if (nst >= std::min(want, cap)) {
        pl.nst = nst;
        pl.ctas_per_sm = k;
        break;
      }
    }
  }
  if (pl.nst < 2) return fail("stage of %d bytes does not fit shared memory", pl.stage_bytes);
  pl.head_bytes = pl.nst * pl.stage_bytes;
  pl.misc_bytes = fixed;
  pl.ring_off = kCtlBytes;
  // the ring region also holds each warp's staged drafts (8 K rows and 8 V
  // rows of bf16, 16 (D + DV) bytes) after streaming
  const int rings = std::max(pl.HC * pl.head_bytes, pl.nwc * 16 * static_cast<int>(D + DV));
  pl.misc_off = pl.ring_off + rings;
  pl.smem = static_cast<size_t>(pl.misc_off) + static_cast<size_t>(pl.nwc) * pl.misc_bytes;
  if (pl.smem > static_cast<size_t>(kSmemPerCTAMax)) return fail("shared memory plan of %zu bytes too large", pl.smem);
  return true;
}

// The tensor-memory streams (vtc_kernel, vtr_kernel) serve head_dim 256 with
// at most 32 packed query rows per KV head; by default (mode 3) the rows-on-M
// one takes the calls where it measured faster (total_tokens: prefix tokens
// from static shapes).
bool tc_eligible(long long h_q, long long h_kv, long long D, long long L, long long total_tokens, bool fp8) {
  if (g_tc == 0 || D != 256 || h_kv <= 0 || h_q % h_kv != 0) return false;
  const long long R = (h_q / h_kv) * L;
  if (R > 32) return false;
  if (g_tc != 3) return true;
  const long long work = total_tokens * h_kv;
  if (work > kSplit256MaxWork) return false;
  return fp8 ? (R > 16 || work < kRowsMR16EndE4m3) : (R <= 16 || work < kRowsMEndBf16);
}

// Plan fields of a two-launch call (tensor-memory or column-split stream,
// then the combine kernel): one KV head per segment, RM = 16 or 32 packed
// rows (MT = RM / 16 tiles).  The stream kernel sets its own launch shape.
bool make_tc_plan(long long h_q, long long h_kv, long long D, long long L, bool fp8, Plan& pl) {
  if (h_kv <= 0 || h_q % h_kv != 0) return fail("h_q (%lld) must be a positive multiple of h_kv (%lld)", h_q, h_kv);
  const long long R = (h_q / h_kv) * L;
  if (R > 32) return fail("packed rows %lld exceed 32", R);
  pl.gq = static_cast<int>(h_q / h_kv);
  pl.R = static_cast<int>(R);
  pl.MT = R <= 16 ? 1 : 2;
  pl.MTW = 1;
  pl.HC = 1;
  pl.n_hg = static_cast<int>(h_kv);
  pl.nwc = pl.MT;
  pl.threads = pl.nwc * 32;
  pl.ek = fp8 ? 1 : 2;
  pl.stage_bytes = 0;
  pl.nst = 0;
  pl.ring_off = kCtlBytes;
  pl.head_bytes = 0;
  pl.misc_bytes = 0;
  pl.misc_off = kCtlBytes + pl.nwc * 32 * static_cast<int>(D);
  pl.smem = static_cast<size_t>(pl.misc_off);
  pl.ctas_per_sm = 1;
  return true;
}

// Column-split stream (vsk_kernel<256, ., 1, false, 2>): head_dim 256 with at
// most 32 packed rows per KV head.  The workspace / epilogue plan is the
// tensor-memory one (one KV head per segment, MT = RM / 16, the epilogue in
// MT warps); the stream runs 2 MT warps per CTA, three CTAs per SM.  Lighter
// warps and more CTAs shorten small calls; from kColSplitEndBf16 (bf16) or
// kColSplitEndE4m3 (e4m3) prefix tokens x KV heads (static shapes) the
// stream-only one-tile kernel with the combine launch measured faster, so by
// default only smaller calls take it.
long long col_split_end(bool fp8) { return fp8 ? kColSplitEndE4m3 : kColSplitEndBf16; }
bool cs_eligible(long long h_q, long long h_kv, long long D, long long L, long long total_tokens, bool fp8) {
  if (g_cs == 0 || D != 256 || h_kv <= 0 || h_q % h_kv != 0 || (h_q / h_kv) * L > 32) return false;
  return g_cs == 2 || total_tokens * h_kv < col_split_end(fp8);
}
// Column-split stream with both 16-row tiles in each warp of the pair
// (vsk_kernel<256, ., 2, 2>): head_dim 256 with 17 to 32 packed rows per KV
// head.  Each K / V element is converted (e4m3 pools) and loaded from shared
// memory once per head instead of once per tile, at the price of the pair's
// score exchange each stage.  It beat the one-tile split on mid-size e4m3
// calls, but the stream-only one-tile kernel with the combine launch
// measured faster still there, so only mode 2 takes it.
bool cs2_eligible(long long h_q, long long h_kv, long long D, long long L) {
  if (g_cs2 != 2 || D != 256 || h_kv <= 0 || h_q % h_kv != 0) return false;
  const long long R = (h_q / h_kv) * L;
  return R > 16 && R <= 32;
}
// Stream-only vsk_kernel then the combine kernel, for calls with at most
// cmb::kMaxL drafts: small and mid-size calls, where the one-launch kernel's
// tail (tickets, a two-level fold of the pieces, the draft block) is a chain
// of memory round trips that the combine launch shortens (the smallest ones
// with the combine launch as a programmatic dependent).  Not, at head_dim 64
// / 128, for long batches, where the one-launch kernel's finishers hide its
// tail behind other CTAs' streaming; at head_dim 256 it measured faster up to
// the 64-sequence batches (from where the column split stops; capped at
// kSplit256MaxWork).  Warps take two tiles (more than 16 packed rows, head_dim
// 64 / 128) from kSplitTwoTileMinTokens prefix tokens.
bool sl_eligible(long long h_q, long long h_kv, long long D, long long L, long long total_tokens, bool fp8) {
  if (g_sl == 0 || (D != 64 && D != 128 && D != 256) || h_kv <= 0 || h_q % h_kv != 0 || L > cmb::kMaxL) return false;
  if (g_sl == 2) return true;
  const long long work = total_tokens * h_kv;
  if (D == 256) {
    // measured for at most 32 packed rows (more stay on the one-launch kernel)
    if ((h_q / h_kv) * L > 32) return false;
    return (g_cs == 0 || work >= col_split_end(fp8)) && work <= kSplit256MaxWork;
  }
  const long long cap = (h_q / h_kv) * L <= 16 ? kSplitLaunchMaxWork16 : kSplitLaunchMaxWork;
  return work <= cap;
}
// Cluster form (one launch: one thread-block cluster per (sequence, KV head)
// segment streams it, then folds its pieces, adds the draft block and writes
// o after a cluster barrier; no tickets, no second launch): small calls,
// where the latency of the other forms' chains of launches and memory round
// trips is what the call costs.  At most cmb::kMaxL drafts, head_dim ==
// v_head_dim, from static shapes.
bool cl_eligible(long long B, long long h_q, long long h_kv, long long D, long long DV, long long L,
                 long long total_tokens) {
  if (g_cl == 0 || D != DV || h_kv <= 0 || h_q % h_kv != 0 || L > cmb::kMaxL || B * h_kv > kClMaxSeg) return false;
  if (D == 256 && (h_q / h_kv) * L > 32) return false;  // head_dim 256 streams by column split: <= 32 rows
  return g_cl == 2 || total_tokens * h_kv <= kClMaxWork;
}

struct StreamPlan {
  int threads, nst, ring_off, head_bytes, misc_off, misc_bytes, per_sm;
  size_t smem;
};
bool make_cs_stream_plan(const Plan& pl, long long D, bool fp8, StreamPlan& sp) {
  const int nwc = 2 * pl.MT;
  sp.threads = nwc * 32;
  sp.per_sm = 3;
  const int stage_bytes = 2 * kStageTokens * static_cast<int>(D) * (fp8 ? 1 : 2);
  // per warp: index ring, mask ring, query tile (e4m3 pools: 16 rows x D/2 f16), score exchange buffer (2 x 1 KB)
  sp.misc_bytes = kIdxRing * 128 + 128 + (fp8 ? 16 * static_cast<int>(D / 2) * 2 : 0) + 2048;
  const int budget = std::min(kSmemPerCTAMax, kSmemPerSM / sp.per_sm - kReservedPerCTA);
  sp.nst = std::min(kMaxStages, (budget - kCtlBytes - nwc * sp.misc_bytes) / stage_bytes);
  if (g_max_stages > 0) sp.nst = std::min(sp.nst, g_max_stages);
  if (sp.nst < 2) return fail("column-split stage of %d bytes does not fit shared memory", stage_bytes);
  sp.ring_off = kCtlBytes;
  sp.head_bytes = sp.nst * stage_bytes;
  sp.misc_off = sp.ring_off + sp.head_bytes;
  sp.smem = static_cast<size_t>(sp.misc_off) + static_cast<size_t>(nwc) * sp.misc_bytes;
  return true;
}

// Two-tile column split: one warp pair per CTA (both tiles of one KV head),
// four CTAs per SM (three if the ring would be shallower than 3 stages).
bool make_cs2_stream_plan(const Plan& pl, long long D, bool fp8, StreamPlan& sp) {
  if (pl.MT != 2) return fail("two-tile column split needs two 16-row tiles (got %d)", pl.MT);
  const int nwc = 2;
  sp.threads = nwc * 32;
  const int stage_bytes = 2 * kStageTokens * static_cast<int>(D) * (fp8 ? 1 : 2);
  // per warp: index ring, mask ring, both query tiles (16 rows x D/2, f16 / bf16),
  // score exchange buffer (2 stage parities x 2 tiles x 1 KB)
  sp.misc_bytes = kIdxRing * 128 + 128 + 2 * 16 * static_cast<int>(D / 2) * 2 + 2 * 2 * 1024;
  sp.nst = 0;
  for (sp.per_sm = 4; sp.per_sm >= 3; --sp.per_sm) {
    const int budget = std::min(kSmemPerCTAMax, kSmemPerSM / sp.per_sm - kReservedPerCTA);
    sp.nst = std::min(kMaxStages, (budget - kCtlBytes - nwc * sp.misc_bytes) / stage_bytes);
    if (g_max_stages > 0) sp.nst = std::min(sp.nst, g_max_stages);
    if (sp.nst >= 3) break;
  }
  if (sp.nst < 2) return fail("two-tile column-split stage of %d bytes does not fit shared memory", stage_bytes);
  sp.ring_off = kCtlBytes;
  sp.head_bytes = sp.nst * stage_bytes;
  sp.misc_off = sp.ring_off + sp.head_bytes;
  sp.smem = static_cast<size_t>(sp.misc_off) + static_cast<size_t>(nwc) * sp.misc_bytes;
  return true;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace: the error word at offset 0, the partials from offset 256 up,
// and the tickets in the LAST cnt_bytes of the buffer, at least 64 KiB.  The
// tickets' place is then the same for every call on a given buffer whatever
// its shapes (up to 16,384 tickets), so the zero tickets a call leaves are the
// ones the next call finds, and no call's partials reach them.
struct WsLayout {
  size_t lse_off, o_off, cnt_bytes, total;
};

WsLayout ws_layout(long long n_cta, long long B, const Plan& pl, long long DV) {
  WsLayout w;
  const long long segs = B * pl.n_hg;
  const long long slots = n_cta + segs;
  const long long rows = slots * pl.HC * 16LL * pl.MT;
  w.lse_off = 256;
  w.o_off = w.lse_off + align256(4 * static_cast<size_t>(rows));
  w.cnt_bytes = std::max(static_cast<size_t>(kTicketBytes), align256(4 * static_cast<size_t>(segs + slots)));
  w.total = align256(w.o_off + 4 * static_cast<size_t>(rows) * static_cast<size_t>(DV)) + w.cnt_bytes;
  return w;
}



struct DevWs {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::mutex g_ws_mu;
std::vector<DevWs> g_ws;
std::vector<int> g_sms;

int device_sms(int dev) {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  if (static_cast<int>(g_sms.size()) <= dev) g_sms.resize(dev + 1, 0);
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

bool check_3d(const vsk_tensor* t, const char* name) {
  if (!t) return fail("%s is NULL", name);
  if (t->ndim != 3) return fail("%s must be 3-d (got ndim %d)", name, t->ndim);
  for (int i = 0; i < 3; ++i)
    if (t->shape[i] < 0) return fail("%s has a negative extent", name);
  if (t->shape[0] > 0 && t->shape[1] > 0 && t->shape[2] > 1 && t->stride[2] != 1)
    return fail("%s: last dimension must be contiguous", name);
  const long long n = t->shape[0] * t->shape[1] * t->shape[2];
  if (n > 0 && !t->data) return fail("%s: NULL data with %lld elements", name, n);
  return true;
}

bool check_1d(const vsk_tensor* t, const char* name) {
  if (!t) return fail("%s is NULL", name);
  if (t->ndim != 1) return fail("%s must be 1-d (got ndim %d)", name, t->ndim);
  if (t->shape[0] < 0) return fail("%s has a negative extent", name);
  if (t->shape[0] > 1 && t->stride[0] != 1) return fail("%s must be contiguous", name);
  if (t->shape[0] > 0 && !t->data) return fail("%s: NULL data", name);
  return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// can_handle of the "verify_splitkv.py" page plus this build's limits.
bool gate(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve, const vsk_tensor* kb,
          const vsk_tensor* vb, const vsk_tensor* qo, const vsk_tensor* kvp, const vsk_tensor* kvi,
          int is_causal, long long mle, long long sliding_window, int has_sinks, float logit_cap,
          long long xai_len) {
  // features the kernel does not implement
  if (has_sinks) return fail("attention sinks are not supported");
  if (sliding_window > 0) return fail("sliding_window_size > 0 is not supported");
  if (logit_cap > 0.f) return fail("logit_cap > 0 is not supported");
  if (xai_len > 0) return fail("xai_temperature_len > 0 is not supported");
  if (!is_causal) return fail("only causal (topk = 1) verify is supported");
  if (!check_3d(q, "q_extend") || !check_3d(ke, "k_extend") || !check_3d(ve, "v_extend") ||
      !check_3d(kb, "k_buffer") || !check_3d(vb, "v_buffer"))
    return false;
  if (!check_1d(qo, "qo_indptr") || !check_1d(kvp, "kv_indptr") || !check_1d(kvi, "kv_indices")) return false;
  const long long h_q = q->shape[1], h_kv = ke->shape[1];
  if (h_kv == 0 || h_q % h_kv != 0) return fail("h_q (%lld) is not a multiple of h_kv (%lld)", h_q, h_kv);
  if (kb->shape[1] != h_kv || vb->shape[1] != h_kv || ve->shape[1] != h_kv)
    return fail("KV head count mismatch between k_extend, v_extend and the buffers");
  const long long D = q->shape[2], Dv = ve->shape[2];
  if (ke->shape[2] != D || kb->shape[2] != D) return fail("head_dim mismatch between q, k_extend and k_buffer");
  if (vb->shape[2] != Dv) return fail("v_head_dim mismatch between v_extend and v_buffer");
  const long long bs = qo->shape[0] - 1;
  if (bs < 1) return fail("batch size must be >= 1");
  if (kvp->shape[0] != bs + 1) return fail("kv_indptr must have B+1 entries");
  if (mle < 1) return fail("max_len_extend must be >= 1");
  if (q->shape[0] != bs * mle) return fail("ragged extend: q has %lld rows, expected B*max_len_extend = %lld", q->shape[0], bs * mle);
  if (ke->shape[0] != q->shape[0] || ve->shape[0] != q->shape[0]) return fail("k_extend/v_extend rows differ from q_extend");
  if (kb->shape[0] != vb->shape[0]) return fail("k_buffer and v_buffer pools differ in size");
  // this build's limits
  if (D != 64 && D != 128 && D != 256) return fail("head_dim %lld not in {64, 128, 256}", D);
  if (Dv != 64 && Dv != 128 && Dv != 256) return fail("v_head_dim %lld not in {64, 128, 256}", Dv);
  if (q->dtype != VSK_DTYPE_BF16 || ke->dtype != VSK_DTYPE_BF16 || ve->dtype != VSK_DTYPE_BF16)
    return fail("q_extend, k_extend and v_extend must be bf16");
  if (kb->dtype != vb->dtype || (kb->dtype != VSK_DTYPE_BF16 && kb->dtype != VSK_DTYPE_FP8E4M3))
    return fail("k_buffer and v_buffer must both be bf16 or both fp8 e4m3");
  if (qo->dtype != VSK_DTYPE_I32 || kvp->dtype != VSK_DTYPE_I32) return fail("indptr arrays must be int32");
  if (kvi->dtype != VSK_DTYPE_I32 && kvi->dtype != VSK_DTYPE_I64) return fail("kv_indices must be int32 or int64");
  const long long R = (h_q / h_kv) * mle;
  const long long maxR = std::max(D, Dv) > 128 ? 64 : 128;
  if (R > maxR) return fail("(h_q/h_kv)*max_len_extend = %lld exceeds %lld", R, maxR);
  const size_t ek = kb->dtype == VSK_DTYPE_BF16 ? 2 : 1;
  for (const vsk_tensor* t : {kb, vb}) {
    if (!aligned(t->data, 16) || (t->stride[0] * ek) % 16 != 0 || (t->stride[1] * ek) % 16 != 0)
      return fail("K/V pool rows must be 16-byte aligned");
  }
  for (const vsk_tensor* t : {q, ke, ve}) {
    if (!aligned(t->data, 4) || (t->stride[0] % 2) != 0 || (t->stride[1] % 2) != 0)
      return fail("q_extend/k_extend/v_extend must be 4-byte aligned with even strides");
  }
  return true;
}

KernelFn pick_kernel(int D, bool fp8, int mtw, int DV = 0, int nst = 0) {
  if (DV != 0 && DV != D) return mtw == 1 ? kernel_dv(D, DV, fp8) : nullptr;
  switch (D) {
    case 64: return kernel_d64(fp8, mtw, false);
    case 128: return kernel_d128(fp8, mtw, false);
    // pipelined stages (faster for e4m3 pools; measured slower for bf16 ones)
    // need a ring of at least three
    case 256: return mtw == 1 ? kernel_d256(fp8, g_pipe && fp8 && nst >= 3 ? 3 : 0) : nullptr;
    default: return nullptr;
  }
}

KernelFn pick_tc_kernel(bool fp8, int rm) { return kernel_tc(fp8, rm); }

KernelFn pick_cs_kernel(bool fp8) { return kernel_d256(fp8, 1); }

KernelFn pick_so_kernel(int D, bool fp8, int mtw) {
  switch (D) {
    case 64: return kernel_d64(fp8, mtw, true);
    case 128: return kernel_d128(fp8, mtw, true);
    // head_dim 256: one tile per warp, one stage after the other (pipelined
    // stages measured 1.8 % slower in this form, e4m3 at 64 sequences)
    case 256: return mtw == 1 ? kernel_d256(fp8, 5) : nullptr;
    default: return nullptr;
  }
}

KernelFn pick_combine_kernel(int D, bool fp8) { return kernel_combine(D, fp8); }

// Shared memory of one combine unit staging nb pieces a batch.
int combine_smem(int D, int nb) {
  return D == 64 ? cmb::Geo<64>::smem(nb) : D == 128 ? cmb::Geo<128>::smem(nb) : cmb::Geo<256>::smem(nb);
}


// Ring entries and shared memory of vtc_kernel (e4m3 pools: an even number
// of entries, so that V rows always sit in odd entries).
template <bool FP8, int RM>
void tc_smem(int& ne, size_t& smem) {
  using G = tc::Geo<256, FP8, RM>;
  ne = std::min(tc::kMaxNE, (kSmemPerCTAMax - G::ring_off) / G::ENT);
  if (FP8) ne &= ~1;
  smem = static_cast<size_t>(G::ring_off) + static_cast<size_t>(ne) * G::ENT;
}

// Ring of vtr_kernel: tile slots (K rows, then V rows of a 64-key tile) for
// e4m3 pools, alternating K and V entries for bf16 pools; and its shared
// memory.
template <bool FP8>
void tr_smem(int& ne, size_t& smem) {
  using G = tr::Geo<FP8>;
  ne = std::min(tr::kMaxNE, (kSmemPerCTAMax - G::ring_off) / G::RING_UNIT);
  // loaders publish a tile's key mask at most ring tiles + 2 ahead of its reader
  ne = std::min(ne, FP8 ? tr::kMaskRing - 3 : 2 * (tr::kMaskRing - 3));
  smem = static_cast<size_t>(G::ring_off) + static_cast<size_t>(ne) * G::RING_UNIT;
}

int prepare_kernel(KernelFn fn) {
  // the attribute is per function and context; set it before every launch
  // configuration query (cheap, idempotent)
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemPerCTAMax) == cudaSuccess;
}

void* internal_workspace(int dev, size_t need, cudaStream_t stream, size_t* bytes) {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  if (static_cast<int>(g_ws.size()) <= dev) g_ws.resize(dev + 1);
  DevWs& w = g_ws[dev];
  if (w.bytes >= need) {
    *bytes = w.bytes;
    return w.ptr;
  }
  if (w.ptr) {
    cudaStreamSynchronize(stream);
    cudaFree(w.ptr);
    w.ptr = nullptr;
    w.bytes = 0;
  }
  void* p = nullptr;
  if (cudaMalloc(&p, need) != cudaSuccess) return nullptr;
  if (cudaMemset(p, 0, need) != cudaSuccess) {
    cudaFree(p);
    return nullptr;
  }
  w.ptr = p;
  w.bytes = need;
  *bytes = need;
  return p;
}

// device address of the allocation-free entry point's built-in scratch
void* static_scratch(int dev);

}  // namespace vsk

using namespace vsk;

extern "C" {

int vsk_can_handle(const vsk_tensor* q_extend, const vsk_tensor* k_extend, const vsk_tensor* v_extend,
                   const vsk_tensor* k_buffer, const vsk_tensor* v_buffer, const vsk_tensor* qo_indptr,
                   const vsk_tensor* kv_indptr, const vsk_tensor* kv_indices, int is_causal,
                   int64_t max_len_extend, int64_t sliding_window_size, int has_sinks, float logit_cap,
                   int64_t xai_temperature_len) {
  g_err.clear();
  return gate(q_extend, k_extend, v_extend, k_buffer, v_buffer, qo_indptr, kv_indptr, kv_indices, is_causal,
              max_len_extend, sliding_window_size, has_sinks, logit_cap, xai_temperature_len)
             ? 1
             : 0;
}

size_t vsk_workspace_size_for_sms(int num_sms, int64_t max_bs, int64_t h_q, int64_t h_kv, int64_t head_dim,
                                  int64_t v_head_dim, int64_t max_len_extend) {
  if (num_sms <= 0 || max_bs < 1 || max_len_extend < 1) return 0;
  for (const int64_t d : {head_dim, v_head_dim})
    if (d != 64 && d != 128 && d != 256) return 0;
  const long long n_cta = static_cast<long long>(num_sms) * 4;  // bound on CTAs per SM
  size_t need = 0;
  for (int fp8 = 0; fp8 < 2; ++fp8) {
    for (int tiles = 1; tiles <= 2; ++tiles) {
      Plan pl;
      if (!make_plan(h_q, h_kv, head_dim, max_len_extend, fp8 != 0, pl, 0, tiles, v_head_dim)) return 0;
      need = std::max(need, ws_layout(n_cta, max_bs, pl, v_head_dim).total);
    }
  }
  Plan tp;
  if (head_dim == 256 && v_head_dim == 256 && (h_q / h_kv) * max_len_extend <= 32 &&
      make_tc_plan(h_q, h_kv, head_dim, max_len_extend, false, tp))
    need = std::max(need, ws_layout(n_cta, max_bs, tp, head_dim).total);
  return need;
}

size_t vsk_workspace_size(int64_t max_bs, int64_t h_q, int64_t h_kv, int64_t head_dim, int64_t v_head_dim,
                          int64_t max_len_extend) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const int sms = device_sms(dev);
  if (sms <= 0) return 0;
  size_t need = vsk_workspace_size_for_sms(sms, max_bs, h_q, h_kv, head_dim, v_head_dim, max_len_extend);
  if (g_num_ctas > 4 * sms) {
    for (int tiles = 1; tiles <= 2; ++tiles) {
      Plan pl;
      if (make_plan(h_q, h_kv, head_dim, max_len_extend, false, pl, 0, tiles, v_head_dim)) {
        const size_t t = ws_layout(g_num_ctas, max_bs, pl, v_head_dim).total;
        if (t > need) need = t;
      }
    }
    Plan tp;
    if (head_dim == 256 && v_head_dim == 256 && h_kv > 0 && h_q % h_kv == 0 && (h_q / h_kv) * max_len_extend <= 32 &&
        make_tc_plan(h_q, h_kv, head_dim, max_len_extend, false, tp)) {
      const size_t t = ws_layout(g_num_ctas, max_bs, tp, head_dim).total;
      if (t > need) need = t;
    }
  }
  return need;
}

int vsk_workspace_init(void* workspace, size_t bytes, void* stream) {
  g_err.clear();
  if (!workspace || bytes == 0) return 1;
  const cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail("cudaMemsetAsync: %s", cudaGetErrorString(e));
  return 1;
}

int vsk_read_error_flags(void* workspace, void* stream, uint32_t* flags) {
  g_err.clear();
  if (!flags) return fail("flags is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail("cudaStreamSynchronize: %s", cudaGetErrorString(e));
  void* ws = workspace;
  if (!ws || ws == VSK_NOALLOC_SCRATCH) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail("no CUDA device");
    if (ws == VSK_NOALLOC_SCRATCH) {
      ws = static_scratch(dev);
      if (!ws) return 0;
    } else {
      std::lock_guard<std::mutex> lk(g_ws_mu);
      if (static_cast<int>(g_ws.size()) > dev) ws = g_ws[dev].ptr;
    }
  }
  if (!ws) {
    *flags = 0;
    return 1;
  }
  e = cudaMemcpy(flags, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail("cudaMemcpy: %s", cudaGetErrorString(e));
  e = cudaMemset(ws, 0, sizeof(uint32_t));
  if (e != cudaSuccess) return fail("cudaMemset: %s", cudaGetErrorString(e));
  return 1;
}

void vsk_set_tuning(int num_ctas, int min_tokens_per_cta) {
  g_num_ctas = num_ctas > 0 ? num_ctas : 0;
  g_min_tokens = min_tokens_per_cta > 0 ? min_tokens_per_cta : 0;
}

void vsk_set_tuning_tiles(int tiles_per_warp) { g_tiles = tiles_per_warp == 1 || tiles_per_warp == 2 ? tiles_per_warp : 0; }

void vsk_set_tuning_tc(int mode) { g_tc = (mode >= 0 && mode <= 2) ? mode : 3; }

void vsk_set_tuning_colsplit(int mode) { g_cs = (mode == 0 || mode == 2) ? mode : 1; }

void vsk_set_tuning_split_launch(int mode) { g_sl = (mode == 0 || mode == 2) ? mode : 1; }

void vsk_set_tuning_cluster(int mode) { g_cl = (mode == 1 || mode == 2) ? mode : 0; }

void vsk_set_tuning_pdl(int mode) { g_pdl = (mode == 0 || mode == 2) ? mode : 1; }

void vsk_set_tuning_pipe(int mode) { g_pipe = mode == 0 ? 0 : 1; }

void vsk_set_tuning_colsplit2(int mode) { g_cs2 = (mode == 0 || mode == 2) ? mode : 1; }

int vsk_launches_per_call(int64_t batch, int64_t h_q, int64_t h_kv, int64_t head_dim, int64_t max_len_extend,
                          int64_t prefix_tokens) {
  if (batch < 1 || h_kv <= 0 || h_q % h_kv != 0 || max_len_extend < 1 || prefix_tokens < 0) return 0;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return 0;
  const long long tokens = prefix_tokens / batch * batch;  // the entry points' static estimate
  if (!tc_eligible(h_q, h_kv, head_dim, max_len_extend, tokens, false) &&
      cl_eligible(batch, h_q, h_kv, head_dim, head_dim, max_len_extend, tokens))
    return 1;
  // (the pool dtype moves only the boundary between two-launch forms: the
  // bf16 thresholds give the same count)
  return (tc_eligible(h_q, h_kv, head_dim, max_len_extend, tokens, false) || cs2_eligible(h_q, h_kv, head_dim, max_len_extend) ||
          cs_eligible(h_q, h_kv, head_dim, max_len_extend, tokens, false) ||
          sl_eligible(h_q, h_kv, head_dim, max_len_extend, tokens, false))
             ? 2
             : 1;
}

const char* vsk_call_form(int64_t batch, int64_t h_q, int64_t h_kv, int64_t head_dim, int64_t v_head_dim,
                          int64_t max_len_extend, int64_t prefix_tokens, int fp8_pool) {
  if (batch < 1 || h_kv <= 0 || h_q % h_kv != 0 || max_len_extend < 1 || prefix_tokens < 0) return "";
  auto ok = [](int64_t d) { return d == 64 || d == 128 || d == 256; };
  if (!ok(head_dim) || !ok(v_head_dim)) return "";
  if (head_dim != v_head_dim) return "one_launch";
  const long long tokens = prefix_tokens / batch * batch;  // the entry points' static estimate
  const bool fp8 = fp8_pool != 0;
  // the same order as the planner's
  if (tc_eligible(h_q, h_kv, head_dim, max_len_extend, tokens, fp8)) return g_tc == 1 ? "tensor_memory" : "tensor_memory_rows";
  if (cl_eligible(batch, h_q, h_kv, head_dim, head_dim, max_len_extend, tokens)) return "cluster";
  if (cs2_eligible(h_q, h_kv, head_dim, max_len_extend)) return "column_split_two_tiles";
  if (cs_eligible(h_q, h_kv, head_dim, max_len_extend, tokens, fp8)) return "column_split";
  if (sl_eligible(h_q, h_kv, head_dim, max_len_extend, tokens, fp8)) return "stream_only";
  return "one_launch";
}

void vsk_set_tuning_shape(int max_ring_stages, int max_kv_heads_per_cta) {
  g_max_stages = max_ring_stages >= 2 ? max_ring_stages : 0;
  g_max_heads = max_kv_heads_per_cta > 0 ? max_kv_heads_per_cta : 0;
}

const char* vsk_last_error(void) { return g_err.c_str(); }

const char* vsk_version(void) { return VSK_VERSION; }

}  // extern "C"

namespace vsk {
// Everything the launches of one call need, decided from static shapes only
// (no device read): the form (one launch, or a stream then the combine
// kernel), the CTA shape, the kernels, the grid, the share floor and the
// workspace layout.  Every entry point plans a call with plan_call and
// enqueues it with enqueue_call, so the workspace a caller (or the built-in
// scratch of the allocation-free entry point) is checked against is the one
// the kernels use.
struct CallPlan {
  bool use_tc = false, use_cs = false, use_sl = false, use_cl = false, use_cs2 = false;
  int cl = 0, cl_smem = 0;  // cluster form: CTAs per cluster, shared memory of one combine group
  int cmb_nb = 8;           // combine units: pieces staged per batch (two batches in flight)
  bool pdl = false;         // combine kernel launched as a programmatic dependent of the stream
  Plan pl{};
  StreamPlan sp{};
  KernelFn fn = nullptr, fn_comb = nullptr;
  int threads = 0;
  size_t smem = 0;
  long long n_cta = 0, n_comb = 0, w_min = 0;
  WsLayout wl{};
  int dev = 0;
  int D = 0;
};

static int plan_call(long long B, long long h_q, long long h_kv, long long D, long long DV, long long L, bool fp8,
                     long long mean_len, CallPlan& cp) {
  cp.D = static_cast<int>(D);
  // the two-launch forms and the cluster form are built for head_dim == v_head_dim only
  const bool same = D == DV;
  cp.use_tc = same && tc_eligible(h_q, h_kv, D, L, mean_len * B, fp8);
  cp.use_cl = !cp.use_tc && cl_eligible(B, h_q, h_kv, D, DV, L, mean_len * B);
  cp.use_cs2 = same && !cp.use_tc && !cp.use_cl && cs2_eligible(h_q, h_kv, D, L);
  cp.use_cs = same && !cp.use_tc && !cp.use_cl && !cp.use_cs2 && cs_eligible(h_q, h_kv, D, L, mean_len * B, fp8);
  cp.use_sl = same && !cp.use_tc && !cp.use_cl && !cp.use_cs && !cp.use_cs2 &&
              sl_eligible(h_q, h_kv, D, L, mean_len * B, fp8);
  Plan& pl = cp.pl;
  if (cp.use_cl && D == 256) {
    // one KV head per cluster, streamed by the column split (two warps per
    // tile) in two 16-row tiles whatever the packed rows (the second empty at
    // <= 16): all four warps stream, the four the combine takes
    if (!make_tc_plan(h_q, h_kv, D, L, fp8, pl)) return 0;
    pl.MT = 2;
    pl.nwc = 2;
    pl.threads = 64;
    if (!make_cs_stream_plan(pl, D, fp8, cp.sp)) return 0;
  } else if (cp.use_cl) {
    // one KV head per cluster, one 16-row tile per warp
    if (!make_plan(h_q, h_kv, D, L, fp8, pl, mean_len * B, 1, DV, 1)) return 0;
  } else if (cp.use_cs2) {
    if (!make_tc_plan(h_q, h_kv, D, L, fp8, pl) || !make_cs2_stream_plan(pl, D, fp8, cp.sp)) return 0;
  } else if ((cp.use_tc || cp.use_cs)
                 ? !make_tc_plan(h_q, h_kv, D, L, fp8, pl)
                 : !make_plan(h_q, h_kv, D, L, fp8, pl, mean_len * B,
                              cp.use_sl && g_tiles == 0 ? (mean_len * B >= kSplitTwoTileMinTokens ? 2 : 1) : 0, DV)) {
    return 0;
  }
  if (cp.use_cs && !make_cs_stream_plan(pl, D, fp8, cp.sp)) return 0;
  cudaError_t e = cudaGetDevice(&cp.dev);
  if (e != cudaSuccess) return fail("cudaGetDevice: %s", cudaGetErrorString(e));
  const int sms = device_sms(cp.dev);
  if (sms <= 0) return fail("cannot query the SM count of device %d", cp.dev);
  // the streaming kernel (the whole call on the one-launch path; the prefix
  // stream on the two-launch paths, followed by the combine kernel)
  cp.threads = pl.threads;
  cp.smem = pl.smem;
  int per_sm = pl.ctas_per_sm;
  if (cp.use_tc) {
    const int rm = 16 * pl.MT;
    const bool rows_m = g_tc != 1;  // the rows-on-M stream (vtr_kernel), else vtc_kernel
    cp.fn = rows_m ? kernel_tr(fp8, rm) : pick_tc_kernel(fp8, rm);
    cp.fn_comb = pick_combine_kernel(256, fp8);
    if (!prepare_kernel(cp.fn) || !prepare_kernel(cp.fn_comb)) return fail("tensor-memory kernels unavailable");
    int ne = 0;
    if (rows_m)
      fp8 ? tr_smem<true>(ne, cp.smem) : tr_smem<false>(ne, cp.smem);
    else if (fp8)
      rm == 16 ? tc_smem<true, 16>(ne, cp.smem) : tc_smem<true, 32>(ne, cp.smem);
    else
      rm == 16 ? tc_smem<false, 16>(ne, cp.smem) : tc_smem<false, 32>(ne, cp.smem);
    if (ne < (rows_m && fp8 ? 2 : 4)) return fail("tensor-memory ring of %d entries is too shallow", ne);
    pl.nst = ne;
    cp.threads = rows_m ? tr::kThreads : tc::kThreads;
  } else if (cp.use_cs || cp.use_cs2) {
    cp.fn = cp.use_cs2 ? kernel_d256(fp8, 4) : pick_cs_kernel(fp8);
    cp.fn_comb = pick_combine_kernel(256, fp8);
    if (!cp.fn || !prepare_kernel(cp.fn) || !prepare_kernel(cp.fn_comb)) return fail("column-split kernels unavailable");
    cp.threads = cp.sp.threads;
    cp.smem = cp.sp.smem;
    per_sm = cp.sp.per_sm;
  } else if (cp.use_cl) {
    cp.fn = D == 64 ? kernel_d64(fp8, 1, true, true) : D == 128 ? kernel_d128(fp8, 1, true, true) : kernel_d256(fp8, 2);
    if (!cp.fn || !prepare_kernel(cp.fn)) return fail("cluster-form kernel for head_dim %lld unavailable", D);
    // at least one 128-thread combine group; the ring region is reused as the
    // groups' shared memory after streaming
    const int nw = D == 256 ? cp.sp.threads / 32 : pl.nwc;  // streaming warps
    const int groups = std::max(nw, 4) / 4;
    cp.threads = groups * cmb::kThreads;
    const long long n_seg = B * pl.n_hg;
    long long c = (mean_len + kClTokensPerCta - 1) / kClTokensPerCta;
    c = std::max(1LL, std::min<long long>(c, kClMax));
    while (c > 1 && n_seg * c > 4LL * sms) --c;  // the workspace bound: at most 4 CTAs per SM
    // a segment's pieces are the cluster's CTAs: two batches of ceil(c / 2)
    // hold them all (the checks below only lower c)
    cp.cmb_nb = static_cast<int>((c + 1) / 2);
    cp.cl_smem = (combine_smem(static_cast<int>(D), cp.cmb_nb) + 127) & ~127;
    // every warp of the CTA (streaming or not) has its index / mask / query region
    const size_t misc_end = D == 256 ? static_cast<size_t>(cp.sp.misc_off) + 4 * groups * cp.sp.misc_bytes
                                     : static_cast<size_t>(pl.misc_off) + 4 * groups * pl.misc_bytes;
    cp.smem = std::max({D == 256 ? cp.sp.smem : cp.smem, misc_end, static_cast<size_t>(groups) * cp.cl_smem});
    if (cp.smem > static_cast<size_t>(kSmemPerCTAMax)) return fail("cluster-form shared memory plan too large");
    if (c > 8 && cudaFuncSetAttribute(reinterpret_cast<const void*>(cp.fn),
                                      cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      c = 8;
    for (;; c = c > 8 ? 8 : c - 1) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = static_cast<unsigned>(c);
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(static_cast<unsigned>(c));
      cfg.blockDim = dim3(cp.threads);
      cfg.dynamicSmemBytes = cp.smem;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int ncl = 0;
      const cudaError_t ce = cudaOccupancyMaxActiveClusters(&ncl, reinterpret_cast<const void*>(cp.fn), &cfg);
      if (ce == cudaSuccess && ncl >= 1) break;
      cudaGetLastError();  // clear the error the query left
      if (c == 1) return fail("cluster-form kernel does not fit (%s)", cudaGetErrorString(ce));
    }
    cp.cl = static_cast<int>(c);
  } else if (cp.use_sl) {
    cp.fn = pick_so_kernel(static_cast<int>(D), fp8, pl.MTW);
    cp.fn_comb = pick_combine_kernel(static_cast<int>(D), fp8);
    if (!cp.fn || !cp.fn_comb || !prepare_kernel(cp.fn) || !prepare_kernel(cp.fn_comb))
      return fail("stream-only kernels for head_dim %lld unavailable", D);
  } else {
    cp.fn = pick_kernel(static_cast<int>(D), fp8, pl.MTW, static_cast<int>(DV), pl.nst);
    if (!cp.fn || !prepare_kernel(cp.fn))
      return fail("kernel for head_dim %lld, v_head_dim %lld unavailable", D, DV);
  }
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, reinterpret_cast<const void*>(cp.fn), cp.threads, cp.smem);
  if (e != cudaSuccess || occ < 1) return fail("kernel does not fit an SM (%s)", cudaGetErrorString(e));
  per_sm = std::min(occ, per_sm);
  cp.n_cta = cp.use_cl ? B * pl.n_hg * cp.cl : g_num_ctas > 0 ? g_num_ctas : static_cast<long long>(sms) * per_sm;
  cp.wl = ws_layout(cp.n_cta, B, pl, DV);
  if (cp.fn_comb) {
    // one combine CTA per (segment, 16-row tile, 32-column slice)
    cp.n_comb = B * pl.n_hg * pl.HC * pl.MT * (D / cmb::kCols);
    if (cp.n_comb > 0x7FFFFFFFLL) return fail("combine grid of %lld CTAs too large", cp.n_comb);
    // pieces in flight per CTA against CTAs per SM: a grid of at most two
    // CTAs per SM stages 2 x 16 pieces (two CTAs fit an SM), up to three
    // CTAs per SM 2 x 8, larger grids 2 x 4
    cp.cmb_nb = cp.n_comb <= 2LL * sms ? 16 : cp.n_comb <= 3LL * sms ? 8 : 4;
    // small calls: the combine kernel's CTAs start while the stream ends (about
    // one microsecond less per call); on mid-size calls that measured neutral
    // to slower, so only up to kPdlMaxWork prefix tokens x KV heads
    cp.pdl = g_pdl == 2 || (g_pdl == 1 && mean_len * B * h_kv <= kPdlMaxWork);
  }
  // Smallest CTA share, from static shapes only (no device read, graph
  // safe): at least 64 tokens and, for small batches where the shares get
  // short, at least the mean prefix / 24 in whole stages, which bounds the
  // pieces a segment's finisher merges.  The two-launch forms (partials
  // folded by the combine launch) do best with every CTA busy: mean prefix / 48.
  if (g_min_tokens > 0) {
    cp.w_min = g_min_tokens;
  } else {
    const long long per =
        (cp.use_cs || cp.use_cs2 || cp.use_sl || cp.use_cl) ? kPiecesPerSegmentColSplit : kPiecesPerSegment;
    const long long wp = (mean_len / per + kStageTokens - 1) / kStageTokens * kStageTokens;
    cp.w_min = std::max(kDefaultMinTokens, wp);
  }
  return 1;
}

// Fills the plan-dependent fields of p and enqueues the call's launches on
// st, with ws (ws_bytes bytes, 256-byte aligned, at least cp.wl.total) as the
// workspace.  Tickets sit in the last cp.wl.cnt_bytes of the buffer; the
// one-launch kernel leaves every ticket it draws at zero, so the last
// kTicketBytes of a buffer are zero between calls, but a call whose ticket
// region is larger (very large batches) first clears the part beyond them,
// where an earlier call may have left partials.
static int enqueue_call(Params& p, const CallPlan& cp, long long B, long long L, unsigned char* ws, size_t ws_bytes,
                        cudaStream_t st) {
  const Plan& pl = cp.pl;
  p.B = static_cast<int>(B);
  p.L = static_cast<int>(L);
  p.gq = pl.gq;
  p.R = pl.R;
  p.HC = pl.HC;
  p.MT = pl.MT;
  p.n_hg = pl.n_hg;
  p.nwc = pl.nwc;
  p.nst = pl.nst;
  p.ring_off = pl.ring_off;
  p.head_bytes = pl.head_bytes;
  p.misc_off = pl.misc_off;
  p.misc_bytes = pl.misc_bytes;
  p.w_min = cp.w_min;
  const size_t cnt_off = (ws_bytes & ~static_cast<size_t>(255)) - cp.wl.cnt_bytes;
  p.err = reinterpret_cast<unsigned*>(ws);
  p.cnt = reinterpret_cast<int*>(ws + cnt_off);
  p.nseg = B * pl.n_hg;
  p.plse = reinterpret_cast<float*>(ws + cp.wl.lse_off);
  p.po = reinterpret_cast<float*>(ws + cp.wl.o_off);
  p.n_stream = static_cast<int>(cp.n_cta);
  p.cl = cp.use_cl ? cp.cl : 0;
  p.cl_smem = cp.cl_smem;
  p.cmb_nb = cp.cmb_nb;
  if (cp.use_cs || cp.use_cs2 || (cp.use_cl && cp.D == 256)) {  // the column-split streams
    p.nwc = cp.sp.threads / 32;
    p.nst = cp.sp.nst;
    p.ring_off = cp.sp.ring_off;
    p.head_bytes = cp.sp.head_bytes;
    p.misc_off = cp.sp.misc_off;
    p.misc_bytes = cp.sp.misc_bytes;
  }
  cudaError_t e;
  if (!cp.fn_comb && cp.wl.cnt_bytes > static_cast<size_t>(kTicketBytes)) {
    e = cudaMemsetAsync(ws + cnt_off, 0, cp.wl.cnt_bytes - kTicketBytes, st);
    if (e != cudaSuccess) return fail("cudaMemsetAsync of the ticket region: %s", cudaGetErrorString(e));
  }
  void* args[] = {&p};
  if (cp.use_cl) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = static_cast<unsigned>(cp.cl);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(cp.n_cta));
    cfg.blockDim = dim3(cp.threads);
    cfg.dynamicSmemBytes = cp.smem;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(cp.fn), args);
  } else {
    e = cudaLaunchKernel(reinterpret_cast<const void*>(cp.fn), dim3(static_cast<unsigned>(cp.n_cta)), dim3(cp.threads),
                         args, cp.smem, st);
  }
  if (e != cudaSuccess) return fail("kernel launch failed: %s", cudaGetErrorString(e));
  if (cp.fn_comb) {
    // the share floor and n_stream let the combine kernel find the pieces the
    // stream launch wrote.  Small calls (cp.pdl) launch it as a programmatic
    // dependent of the stream: its CTAs may start (and read the call's
    // lengths) before the stream ends, and wait for it before reading anything
    // it wrote.
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(cp.n_comb));
    cfg.blockDim = dim3(cmb::kThreads);
    cfg.dynamicSmemBytes = combine_smem(cp.D, cp.cmb_nb);
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = cp.pdl ? 1 : 0;
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(cp.fn_comb), args);
    if (e != cudaSuccess) return fail("combine kernel launch failed: %s", cudaGetErrorString(e));
  }
  return 1;
}

// Plans the call, resolves the workspace (NULL: the library-owned per-device
// buffer) and enqueues the launches.
static int launch_with_plan(Params& p, long long B, long long h_q, long long h_kv, long long D, long long DV, long long L,
                            bool fp8, void* workspace, size_t workspace_bytes, void* stream, long long mean_len) {
  CallPlan cp;
  if (!plan_call(B, h_q, h_kv, D, DV, L, fp8, mean_len, cp)) return 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  size_t ws_bytes = workspace_bytes;
  if (!ws) {
    ws = static_cast<unsigned char*>(internal_workspace(cp.dev, cp.wl.total, st, &ws_bytes));
    if (!ws) return fail("cannot allocate a %zu-byte workspace", cp.wl.total);
  } else if (workspace_bytes < cp.wl.total) {
    return fail("workspace of %zu bytes is smaller than the %zu bytes needed", workspace_bytes, cp.wl.total);
  } else if (!aligned(ws, 256)) {
    return fail("workspace must be 256-byte aligned");
  }
  return enqueue_call(p, cp, B, L, ws, ws_bytes, st);
}

// The checks and the parameter block shared by the flat entry points (causal,
// tree, fused store, allocation-free); cm / mi select tree verify (both null:
// causal drafts), ocl the fused store.  Returns the static shapes the plan
// needs.
struct CallShape {
  long long B, h_q, h_kv, D, DV, L, mean_len;
  bool fp8;
};

static int prepare_verify(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve, const vsk_tensor* o,
                          const vsk_tensor* kb, const vsk_tensor* vb, const vsk_tensor* qo, const vsk_tensor* kvp,
                          const vsk_tensor* kvi, int is_causal, int64_t max_len_extend, float k_scale, float v_scale,
                          float sm_scale, const vsk_tensor* cm, const vsk_tensor* mi, const vsk_tensor* ocl, Params& p,
                          CallShape& cs) {
  if (!gate(q, ke, ve, kb, vb, qo, kvp, kvi, is_causal, max_len_extend, -1, 0, 0.f, -1)) return 0;
  if (!check_3d(o, "o_extend")) return 0;
  if (o->dtype != VSK_DTYPE_BF16 || o->shape[0] != q->shape[0] || o->shape[1] != q->shape[1] ||
      o->shape[2] != ve->shape[2])
    return fail("o_extend must be bf16 [B*l_ext, h_q, v_head_dim]");
  if (!aligned(o->data, 4) || (o->stride[0] % 2) != 0 || (o->stride[1] % 2) != 0)
    return fail("o_extend must be 4-byte aligned with even strides");
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale)) return fail("k_scale and v_scale must be finite");

  memset(&p, 0, sizeof p);
  p.q = static_cast<const __nv_bfloat16*>(q->data);
  p.q_s0 = q->stride[0];
  p.q_s1 = q->stride[1];
  p.ke = static_cast<const __nv_bfloat16*>(ke->data);
  p.ke_s0 = ke->stride[0];
  p.ke_s1 = ke->stride[1];
  p.ve = static_cast<const __nv_bfloat16*>(ve->data);
  p.ve_s0 = ve->stride[0];
  p.ve_s1 = ve->stride[1];
  p.o = static_cast<__nv_bfloat16*>(const_cast<void*>(o->data));
  p.o_s0 = o->stride[0];
  p.o_s1 = o->stride[1];
  p.kb = static_cast<const unsigned char*>(kb->data);
  const int ek = kb->dtype == VSK_DTYPE_FP8E4M3 ? 1 : 2;
  p.kb_s0 = kb->stride[0] * ek;
  p.kb_s1 = kb->stride[1] * ek;
  p.vb = static_cast<const unsigned char*>(vb->data);
  p.vb_s0 = vb->stride[0] * ek;
  p.vb_s1 = vb->stride[1] * ek;
  p.qo = static_cast<const int*>(qo->data);
  p.kvp = static_cast<const int*>(kvp->data);
  p.kvi = kvi->data;
  p.idx64 = kvi->dtype == VSK_DTYPE_I64;
  p.n_idx = kvi->shape[0];
  p.pool = kb->shape[0];
  p.n_rows = q->shape[0];
  const long long D = q->shape[2];
  const double sm = (sm_scale > 0.f && std::isfinite(sm_scale)) ? static_cast<double>(sm_scale)
                                                                 : 1.0 / std::sqrt(static_cast<double>(D));
  const double log2e = 1.4426950408889634;
  p.scale2 = static_cast<float>(sm * static_cast<double>(k_scale) * log2e);
  p.dscale2 = static_cast<float>(sm * log2e);
  p.dvs = 1.f;
  p.v_scale = v_scale;
  p.cmask = cm ? static_cast<const unsigned char*>(cm->data) : nullptr;
  p.mindptr = mi ? mi->data : nullptr;
  p.mindptr64 = (mi && mi->dtype == VSK_DTYPE_I64) ? 1 : 0;
  p.n_mask = cm ? cm->shape[0] : 0;
  if (p.cmask == nullptr) p.mindptr = nullptr;
  if (ocl) {
    if (!check_1d(ocl, "out_cache_loc")) return 0;
    if (ocl->dtype != VSK_DTYPE_I32 && ocl->dtype != VSK_DTYPE_I64) return fail("out_cache_loc must be int32 or int64");
    if (ocl->shape[0] != q->shape[0]) return fail("out_cache_loc must have one entry per q_extend row");
    if (!(k_scale > 0.f) || !(v_scale > 0.f)) return fail("storing into the cache needs k_scale > 0 and v_scale > 0");
    p.wmode = 1;
    p.ocl = ocl->data;
    p.ocl64 = ocl->dtype == VSK_DTYPE_I64;
    p.kw = static_cast<unsigned char*>(const_cast<void*>(kb->data));
    p.vw = static_cast<unsigned char*>(const_cast<void*>(vb->data));
    p.kq = k_scale;
    p.vq = v_scale;
  }
  cs.B = qo->shape[0] - 1;
  cs.h_q = q->shape[1];
  cs.h_kv = ke->shape[1];
  cs.D = D;
  cs.DV = ve->shape[2];
  cs.L = max_len_extend;
  cs.fp8 = kb->dtype == VSK_DTYPE_FP8E4M3;
  cs.mean_len = kvi->shape[0] / cs.B;
  return 1;
}

// Shared body of the workspace entry points.
static int run_verify(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve, const vsk_tensor* o,
                      const vsk_tensor* kb, const vsk_tensor* vb, const vsk_tensor* qo, const vsk_tensor* kvp,
                      const vsk_tensor* kvi, int is_causal, int64_t max_len_extend, float k_scale, float v_scale,
                      float sm_scale, void* workspace, size_t workspace_bytes, void* stream, const vsk_tensor* cm,
                      const vsk_tensor* mi, const vsk_tensor* ocl = nullptr) {
  Params p;
  CallShape cs;
  if (!prepare_verify(q, ke, ve, o, kb, vb, qo, kvp, kvi, is_causal, max_len_extend, k_scale, v_scale, sm_scale, cm,
                      mi, ocl, p, cs))
    return 0;
  return launch_with_plan(p, cs.B, cs.h_q, cs.h_kv, cs.D, cs.DV, cs.L, cs.fp8, workspace, workspace_bytes, stream,
                          cs.mean_len);
}

bool check_2d(const vsk_tensor* t, const char* name) {
  if (!t) return fail("%s is NULL", name);
  if (t->ndim != 2) return fail("%s must be 2-d (got ndim %d)", name, t->ndim);
  if (t->shape[0] < 0 || t->shape[1] < 0) return fail("%s has a negative extent", name);
  if (t->shape[0] > 0 && t->shape[1] > 1 && t->stride[1] != 1) return fail("%s: rows must be contiguous", name);
  if (t->shape[0] * t->shape[1] > 0 && !t->data) return fail("%s: NULL data", name);
  return true;
}

// Drafts already written to a paged cache (the unified verify of the
// "aiter_backend.py" page): sequence b's cache position t lives in pool row
// block_table[b][t / page_size] * page_size + t % page_size, its prefix is
// positions [0, seq_lens[b]) and its drafts [seq_lens[b], seq_lens[b] + L).
static int run_paged(const vsk_tensor* q, const vsk_tensor* o, const vsk_tensor* kc, const vsk_tensor* vc,
                     const vsk_tensor* bt, const vsk_tensor* sl, int64_t page_size, int64_t mle, float k_scale,
                     float v_scale, float sm_scale, void* workspace, size_t workspace_bytes, void* stream,
                     const vsk_tensor* k_new = nullptr, const vsk_tensor* v_new = nullptr) {
  if (!check_3d(q, "q") || !check_3d(o, "o") || !check_3d(kc, "k_cache") || !check_3d(vc, "v_cache")) return 0;
  if (!check_2d(bt, "block_table") || !check_1d(sl, "seq_lens")) return 0;
  if (page_size < 1) return fail("page_size must be >= 1");
  if (mle < 1) return fail("max_len_extend must be >= 1");
  const long long bs = sl->shape[0];
  if (bs < 1) return fail("batch size must be >= 1");
  if (bt->shape[0] != bs) return fail("block_table must have one row per sequence (B = %lld)", bs);
  if (bt->shape[1] < 1) return fail("block_table has no columns");
  if (bt->shape[1] * page_size > INT_MAX) return fail("block_table columns x page_size exceeds 2^31 - 1");
  if (bt->shape[1] * page_size < mle) return fail("block_table covers fewer than max_len_extend positions");
  if (bt->dtype != VSK_DTYPE_I32 || sl->dtype != VSK_DTYPE_I32) return fail("block_table and seq_lens must be int32");
  if (q->shape[0] != bs * mle)
    return fail("ragged extend: q has %lld rows, expected B*max_len_extend = %lld", q->shape[0], bs * mle);
  const long long h_q = q->shape[1], h_kv = kc->shape[1], D = q->shape[2];
  if (h_kv == 0 || h_q % h_kv != 0) return fail("h_q (%lld) is not a multiple of h_kv (%lld)", h_q, h_kv);
  if (vc->shape[1] != h_kv) return fail("KV head count mismatch between k_cache and v_cache");
  const long long DV = vc->shape[2];
  if (kc->shape[2] != D) return fail("head_dim mismatch between q and k_cache");
  if (D != 64 && D != 128 && D != 256) return fail("head_dim %lld not in {64, 128, 256}", D);
  if (DV != 64 && DV != 128 && DV != 256) return fail("v_head_dim %lld not in {64, 128, 256}", DV);
  if (kc->shape[0] != vc->shape[0]) return fail("k_cache and v_cache pools differ in size");
  if (kc->shape[0] % page_size != 0) return fail("cache rows (%lld) are not a whole number of pages", kc->shape[0]);
  if (q->dtype != VSK_DTYPE_BF16) return fail("q must be bf16");
  if (kc->dtype != vc->dtype || (kc->dtype != VSK_DTYPE_BF16 && kc->dtype != VSK_DTYPE_FP8E4M3))
    return fail("k_cache and v_cache must both be bf16 or both fp8 e4m3");
  const long long R = (h_q / h_kv) * mle;
  const long long maxR = std::max(D, DV) > 128 ? 64 : 128;
  if (R > maxR) return fail("(h_q/h_kv)*max_len_extend = %lld exceeds %lld", R, maxR);
  const size_t ek = kc->dtype == VSK_DTYPE_BF16 ? 2 : 1;
  for (const vsk_tensor* t : {kc, vc}) {
    if (!aligned(t->data, 16) || (t->stride[0] * ek) % 16 != 0 || (t->stride[1] * ek) % 16 != 0)
      return fail("K/V cache rows must be 16-byte aligned");
  }
  if (o->dtype != VSK_DTYPE_BF16 || o->shape[0] != q->shape[0] || o->shape[1] != h_q || o->shape[2] != DV)
    return fail("o must be bf16 [B*l_ext, h_q, v_head_dim]");
  for (const vsk_tensor* t : {q, o}) {
    if (!aligned(t->data, 4) || (t->stride[0] % 2) != 0 || (t->stride[1] % 2) != 0)
      return fail("q and o must be 4-byte aligned with even strides");
  }
  if (!aligned(bt->data, 4) || !aligned(sl->data, 4)) return fail("block_table and seq_lens must be 4-byte aligned");
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale)) return fail("k_scale and v_scale must be finite");

  Params p;
  memset(&p, 0, sizeof p);
  p.q = static_cast<const __nv_bfloat16*>(q->data);
  p.q_s0 = q->stride[0];
  p.q_s1 = q->stride[1];
  p.o = static_cast<__nv_bfloat16*>(const_cast<void*>(o->data));
  p.o_s0 = o->stride[0];
  p.o_s1 = o->stride[1];
  p.kb = static_cast<const unsigned char*>(kc->data);
  p.kb_s0 = kc->stride[0] * static_cast<long long>(ek);
  p.kb_s1 = kc->stride[1] * static_cast<long long>(ek);
  p.vb = static_cast<const unsigned char*>(vc->data);
  p.vb_s0 = vc->stride[0] * static_cast<long long>(ek);
  p.vb_s1 = vc->stride[1] * static_cast<long long>(ek);
  p.pool = kc->shape[0];
  p.n_rows = q->shape[0];
  p.paged = 1;
  p.bt = static_cast<const int*>(bt->data);
  p.bt_s0 = bt->stride[0];
  p.bt_cols = static_cast<int>(bt->shape[1]);
  p.page = static_cast<int>(page_size);
  {
    int l = 0;
    while ((1LL << l) < page_size) ++l;
    p.pg_l = l;
    p.pg_m = static_cast<unsigned>(((1ULL << (32 + l)) + static_cast<unsigned long long>(page_size) - 1) /
                                       static_cast<unsigned long long>(page_size) -
                                   (1ULL << 32));
  }
  p.slens = static_cast<const int*>(sl->data);
  const double sm = (sm_scale > 0.f && std::isfinite(sm_scale)) ? static_cast<double>(sm_scale)
                                                                 : 1.0 / std::sqrt(static_cast<double>(D));
  const double log2e = 1.4426950408889634;
  // every cached key, drafts included, carries the cache's scales
  p.scale2 = static_cast<float>(sm * static_cast<double>(k_scale) * log2e);
  p.dscale2 = p.scale2;
  p.dvs = v_scale;
  p.v_scale = v_scale;
  if (k_new || v_new) {
    if (!check_3d(k_new, "k_new") || !check_3d(v_new, "v_new")) return 0;
    if (k_new->dtype != VSK_DTYPE_BF16 || v_new->dtype != VSK_DTYPE_BF16) return fail("k_new and v_new must be bf16");
    if (k_new->shape[0] != q->shape[0] || v_new->shape[0] != q->shape[0] || k_new->shape[1] != h_kv ||
        v_new->shape[1] != h_kv || k_new->shape[2] != D || v_new->shape[2] != DV)
      return fail("k_new / v_new must be [B*l_ext, h_kv, head_dim / v_head_dim]");
    for (const vsk_tensor* t : {k_new, v_new}) {
      if (!aligned(t->data, 4) || (t->stride[0] % 2) != 0 || (t->stride[1] % 2) != 0)
        return fail("k_new and v_new must be 4-byte aligned with even strides");
    }
    if (!(k_scale > 0.f) || !(v_scale > 0.f)) return fail("storing into the cache needs k_scale > 0 and v_scale > 0");
    p.ke = static_cast<const __nv_bfloat16*>(k_new->data);
    p.ke_s0 = k_new->stride[0];
    p.ke_s1 = k_new->stride[1];
    p.ve = static_cast<const __nv_bfloat16*>(v_new->data);
    p.ve_s0 = v_new->stride[0];
    p.ve_s1 = v_new->stride[1];
    p.wmode = 2;
    p.kw = static_cast<unsigned char*>(const_cast<void*>(kc->data));
    p.vw = static_cast<unsigned char*>(const_cast<void*>(vc->data));
    p.kq = k_scale;
    p.vq = v_scale;
  }
  // the block table bounds every sequence's length: its capacity stands in for the mean
  return launch_with_plan(p, bs, h_q, h_kv, D, DV, mle, kc->dtype == VSK_DTYPE_FP8E4M3, workspace, workspace_bytes,
                          stream, bt->shape[1] * page_size);
}
}  // namespace vsk

extern "C" {

int verify_splitkv_paged_fwd(const vsk_tensor* q, const vsk_tensor* o, const vsk_tensor* k_cache,
                             const vsk_tensor* v_cache, const vsk_tensor* block_table, const vsk_tensor* seq_lens,
                             int64_t page_size, int64_t max_len_extend, float k_scale, float v_scale, float sm_scale,
                             void* workspace, size_t workspace_bytes, void* stream) {
  g_err.clear();
  return run_paged(q, o, k_cache, v_cache, block_table, seq_lens, page_size, max_len_extend, k_scale, v_scale,
                   sm_scale, workspace, workspace_bytes, stream);
}

int verify_splitkv_paged_write_fwd(const vsk_tensor* q, const vsk_tensor* k_new, const vsk_tensor* v_new,
                                   const vsk_tensor* o, const vsk_tensor* k_cache, const vsk_tensor* v_cache,
                                   const vsk_tensor* block_table, const vsk_tensor* seq_lens, int64_t page_size,
                                   int64_t max_len_extend, float k_scale, float v_scale, float sm_scale,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  g_err.clear();
  if (!k_new || !v_new) return fail("k_new and v_new are required");
  return run_paged(q, o, k_cache, v_cache, block_table, seq_lens, page_size, max_len_extend, k_scale, v_scale,
                   sm_scale, workspace, workspace_bytes, stream, k_new, v_new);
}

int verify_splitkv_write_fwd(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve, const vsk_tensor* o,
                             const vsk_tensor* kb, const vsk_tensor* vb, const vsk_tensor* qo, const vsk_tensor* kvp,
                             const vsk_tensor* kvi, const vsk_tensor* out_cache_loc, int64_t max_len_extend,
                             float k_scale, float v_scale, float sm_scale, void* workspace, size_t workspace_bytes,
                             void* stream) {
  g_err.clear();
  if (!out_cache_loc) return fail("out_cache_loc is NULL");
  return run_verify(q, ke, ve, o, kb, vb, qo, kvp, kvi, 1, max_len_extend, k_scale, v_scale, sm_scale, workspace,
                    workspace_bytes, stream, nullptr, nullptr, out_cache_loc);
}

int verify_splitkv_fwd(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve, const vsk_tensor* o,
                       const vsk_tensor* kb, const vsk_tensor* vb, const vsk_tensor* qo, const vsk_tensor* kvp,
                       const vsk_tensor* kvi, int is_causal, int64_t max_len_extend, float k_scale, float v_scale,
                       float sm_scale, void* workspace, size_t workspace_bytes, void* stream) {
  g_err.clear();
  return run_verify(q, ke, ve, o, kb, vb, qo, kvp, kvi, is_causal, max_len_extend, k_scale, v_scale, sm_scale,
                    workspace, workspace_bytes, stream, nullptr, nullptr);
}

int verify_splitkv_tree_fwd(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve, const vsk_tensor* o,
                            const vsk_tensor* kb, const vsk_tensor* vb, const vsk_tensor* qo, const vsk_tensor* kvp,
                            const vsk_tensor* kvi, const vsk_tensor* custom_mask, const vsk_tensor* mask_indptr,
                            int64_t max_len_extend, float k_scale, float v_scale, float sm_scale, void* workspace,
                            size_t workspace_bytes, void* stream) {
  g_err.clear();
  if (!check_1d(custom_mask, "custom_mask") || !check_1d(mask_indptr, "mask_indptr")) return 0;
  if (custom_mask->dtype != VSK_DTYPE_U8) return fail("custom_mask must be uint8 (or bool)");
  if (mask_indptr->dtype != VSK_DTYPE_I32 && mask_indptr->dtype != VSK_DTYPE_I64)
    return fail("mask_indptr must be int32 or int64");
  if (!qo || mask_indptr->shape[0] != qo->shape[0]) return fail("mask_indptr must have B+1 entries");
  return run_verify(q, ke, ve, o, kb, vb, qo, kvp, kvi, 1, max_len_extend, k_scale, v_scale, sm_scale, workspace,
                    workspace_bytes, stream, custom_mask, mask_indptr);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot call cudaMalloc at all: engines that hand every free
// byte of HBM to their own pool allocator at start-up and forbid stray device
// allocations (a cudaMalloc there can fail, fragment the pool, or stall every
// stream while the driver maps memory), and plugin hosts whose interface
// passes only input and output pointers with no workspace.  For them the
// scratch this kernel needs (one ticket per segment, the error word and the
// per-CTA log-sum-exp partials) lives in the array below, which the driver
// creates when the library's module is loaded on a GPU and keeps until the
// process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_vsk_static_scratch[VSK_NOALLOC_SCRATCH_BYTES];

namespace vsk {

std::mutex g_static_mu;
std::vector<void*> g_static_addr;  // per device: device address of g_vsk_static_scratch

// Device address of the scratch array on device dev, which must be the
// current device.  The host-side name is only a stand-in, so the address is
// asked from the runtime once per device and cached.
void* static_scratch(int dev) {
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (static_cast<int>(g_static_addr.size()) <= dev) g_static_addr.resize(dev + 1, nullptr);
  if (!g_static_addr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_vsk_static_scratch);
    if (e != cudaSuccess) {
      fail("cudaGetSymbolAddress of the built-in scratch failed: %s", cudaGetErrorString(e));
      return nullptr;
    }
    g_static_addr[dev] = ptr;
  }
  return g_static_addr[dev];
}

}  // namespace vsk

extern "C" int verify_splitkv_fwd_noalloc(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve,
                                          const vsk_tensor* o, const vsk_tensor* kb, const vsk_tensor* vb,
                                          const vsk_tensor* qo, const vsk_tensor* kvp, const vsk_tensor* kvi,
                                          int is_causal, int64_t max_len_extend, float k_scale, float v_scale,
                                          float sm_scale, void* stream) {
  g_err.clear();
  Params p;
  CallShape cs;
  if (!prepare_verify(q, ke, ve, o, kb, vb, qo, kvp, kvi, is_causal, max_len_extend, k_scale, v_scale, sm_scale,
                      nullptr, nullptr, nullptr, p, cs))
    return 0;
  // the same plan (form, grid, workspace layout) verify_splitkv_fwd would use
  CallPlan cp;
  if (!plan_call(cs.B, cs.h_q, cs.h_kv, cs.D, cs.DV, cs.L, cs.fp8, cs.mean_len, cp)) return 0;
  if (cp.wl.total > static_cast<size_t>(VSK_NOALLOC_SCRATCH_BYTES))
    return fail("this problem needs %zu bytes of scratch, more than the %d bytes built into the library for "
                "verify_splitkv_fwd_noalloc; use verify_splitkv_fwd with a caller workspace",
                cp.wl.total, VSK_NOALLOC_SCRATCH_BYTES);
  unsigned char* scratch = static_cast<unsigned char*>(static_scratch(cp.dev));
  if (!scratch) return 0;
  // The array keeps whatever the previous call left: zero the error word and
  // this call's whole ticket span (at the end of the array) before its
  // kernels run.
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(scratch, 0, 256, st);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(scratch + VSK_NOALLOC_SCRATCH_BYTES - cp.wl.cnt_bytes, 0, cp.wl.cnt_bytes, st);
  if (e != cudaSuccess) return fail("cudaMemsetAsync on the built-in scratch: %s", cudaGetErrorString(e));
  return enqueue_call(p, cp, cs.B, cs.L, scratch, VSK_NOALLOC_SCRATCH_BYTES, st);
}
