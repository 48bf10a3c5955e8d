// ---------------------------------------------------------------------------
// Combine kernel of the two-launch forms (the column-split and tensor-memory
// streams at head_dim 256, the stream-only vsk_kernel at 64 / 128).  Split-KV (flash-decode) attention computes one
// (o, log-sum-exp) partial per CTA piece of a sequence's prefix and merges
// them with the log-sum-exp rule; the verify step then continues the same
// softmax over the causal draft-draft block (verify_splitkv.py page,
// `_verify_combine_stage2`: the prefix splits are merged by log-sum-exp, then
// merged again with the causal draft-draft block's scores).
//
// When this kernel starts, the stream launch before it on the same stream has
// written every piece's partial, so no ticket or arrival order is needed: one
// CTA per (segment, KV head of the segment, 16-row query tile, 32-column
// slice of the output) reads the segment's pieces straight away.  Thread t
// owns row t / 8 of the tile and four output columns.  The pieces' 16 x 32
// blocks are staged in shared memory by cp.async, nb pieces a batch with two
// batches in flight (each thread copies the 16 bytes it will fold, each warp
// the log-sum-exps of its four rows, so the fold needs no block barrier), and
// every thread folds its columns with a running maximum and sum.  The CTA
// then computes the draft scores of the tile (each warp a quarter of the head
// dimension, summed in a fixed order), continues the softmax and writes its
// 16 x 32 block of o.  The fused-store forms store the new
// draft rows here too: tile 0's CTAs, each its 32-column slice of every row,
// so every stored element has exactly one writer.
//
// The pieces of segment s = (b, hg) are found the way every kernel of a call
// cuts the work: segments of virtual length max(P_b, 1) laid end to end, CTA
// c of the stream grid (p.n_stream CTAs) owning [c W, c W + W) with
// W = max(ceil(total / n_stream), w_min); piece c of s sits in slot c + s,
// KV head hc of the segment's HC at partial (slot HC + hc).
// ---------------------------------------------------------------------------
namespace cmb {
constexpr int kThreads = 128;              // four warps
constexpr int kCols = 32;                  // output columns per CTA
constexpr int kMaxL = 32;                  // draft keys served
constexpr int kScPitch = kMaxL + 1;
constexpr int kPieceBytes = 16 * kCols * 4;  // one piece's staged 16 x 32 fp32 block
constexpr int kPieceLseBytes = 16 * 4;       // ... and its 16 log-sum-exps
constexpr int kBatchMax = 32;                // pieces per batch at most (one log-sum-exp copy per lane)
// Shared-memory map of the head_dim D instance (bytes).
template <int D>
struct Geo {
  static constexpr int kSlices = D / kCols;
  static constexpr int kKPitch = D * 2 + 16;  // staged K row, bf16 (padded: conflict-free fragment reads)
  static constexpr int kScanOff = 0;          // 2 x 4 x i64 block sums
  static constexpr int kSrcOff = 128;         // [kMaxL] i64: row the draft is read from (-1: no row)
  static constexpr int kDstOff = kSrcOff + kMaxL * 8;    // [kMaxL] i64: row it is stored to (-1: none)
  static constexpr int kKOff = kDstOff + kMaxL * 8;      // [kMaxL][kKPitch] draft K rows
  static constexpr int kVOff = kKOff + kMaxL * kKPitch;  // [kMaxL][kCols] bf16 draft V slice
  static constexpr int kScOff = kVOff + kMaxL * kCols * 2;     // per warp [16][kScPitch] partial scores
  static constexpr int kStageOff = (kScOff + 4 * 16 * kScPitch * 4 + 127) & ~127;
  // staged pieces: 2 nb blocks [16][kCols] fp32, then 2 nb x 16 log-sum-exps
  static constexpr int smem(int nb) { return kStageOff + 2 * nb * (kPieceBytes + kPieceLseBytes); }
  static_assert(smem(kBatchMax) <= 227 * 1024, "combine kernel fits an SM");
  static_assert(kKOff % 16 == 0 && kVOff % 16 == 0 && kStageOff % 16 == 0, "16-byte aligned regions");
};
}  // namespace cmb

// One unit of the combine: segment s_idx, KV head hc of the segment, 16-row
// tile `tile`, 32-column slice ch, served by 128 threads (tid 0..127) with
// the shared-memory region smem (Geo<D>::smem(p.cmb_nb) bytes).  CL = false: the
// combine kernel, which finds the segment's pieces by the stream launch's cut
// of the work (a block scan) and synchronises with __syncthreads.  CL = true:
// the cluster form, whose pieces are slot0 .. slot0 + npc - 1 and whose
// threads meet at named barrier `bar` (128 threads).
template <int D, bool FP8, bool CL>
__device__ __forceinline__ void combine_unit(const Params& p, unsigned char* smem, const int tid, const int bar,
                                             const long long s_idx, const int hc, const int tile, const int ch,
                                             long long slot0, long long npc) {
  using namespace cmb;
  using G = Geo<D>;
  constexpr int kKPitch = G::kKPitch;
  constexpr int kScanOff = G::kScanOff, kSrcOff = G::kSrcOff, kDstOff = G::kDstOff, kKOff = G::kKOff;
  constexpr int kVOff = G::kVOff, kScOff = G::kScOff, kStageOff = G::kStageOff;
  constexpr int DW = D / 4;    // head dimensions of one warp's part of the draft scores
  constexpr int KSW = DW / 16;  // its k-steps
  const int lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, j = lane & 3;
  const int RM = 16 * p.MT;
  auto sync = [&]() {
    if constexpr (CL)
      named_bar_sync(bar, kThreads);
    else
      __syncthreads();
  };
  const float NEG_INF = -INFINITY;
  Seg sg;
  sg.b = static_cast<int>(s_idx / p.n_hg);
  sg.hg = static_cast<int>(s_idx % p.n_hg);
  // Every load below depends on the segment index alone: all are issued
  // before any of them is used, so they cost one memory round trip together.
  int qa, qe;  // the sequence's draft rows in q / k_ext / v_ext / o (qo_indptr)
  if (p.qo) {
    qa = __ldg(p.qo + sg.b);
    qe = __ldg(p.qo + sg.b + 1);
  } else {
    qa = sg.b * p.L;
    qe = qa + p.L;
  }
  load_seq(p, sg.b, sg.P, sg.kv0);
  // block sums of the virtual segment lengths: all of them and those before b
  long long* scan = reinterpret_cast<long long*>(smem + kScanOff);
  if constexpr (!CL) {
    long long tot_t = 0, bef_t = 0;
    for (int bb = tid; bb < p.B; bb += kThreads) {
      int P_;
      long long k_;
      seq_info(p, bb, P_, k_);
      const long long ln = max(P_, 1);
      tot_t += ln;
      if (bb < sg.b) bef_t += ln;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tot_t += __shfl_xor_sync(0xffffffffu, tot_t, o);
      bef_t += __shfl_xor_sync(0xffffffffu, bef_t, o);
    }
    if (lane == 0) {
      scan[warp] = tot_t;
      scan[4 + warp] = bef_t;
    }
  }
  sg.len = max(sg.P, 1);
  const int kvh = sg.hg * p.HC + hc;
  const int col0 = ch * kCols;
  const bool writer = tile == 0;  // stores this CTA's column slice of the new drafts
  const bool flagger = tid == 0 && ch == 0 && tile == 0 && hc == 0;
  int s_b;
  {
    const bool ok = qa >= 0 && qe - qa == p.L && static_cast<long long>(qa) + p.L <= p.n_rows;
    if (!ok && flagger) atomicOr(p.err, kErrBadQoIndptr);
    s_b = ok ? qa : sg.b * p.L;
  }
  // per draft key: the row it is read from and the row it is stored to
  long long* ksrc = reinterpret_cast<long long*>(smem + kSrcOff);
  long long* kdst = reinterpret_cast<long long*>(smem + kDstOff);
  if (tid < p.L) {
    const int key = tid;
    long long src = static_cast<long long>(s_b) + key, dst = -1;
    if (p.paged) {
      // drafts at cache positions P + key (the paged store puts them there)
      const long long row = paged_row(p, sg.b, sg.P + key);
      if (row < 0 && writer && ch == 0) atomicOr(p.err, kErrBadIndex);
      if (p.wmode == 2) {
        dst = row;
        if (row < 0) src = -1;
      } else {
        src = row;
      }
    } else if (p.wmode == 1) {
      const long long d = p.ocl64 ? static_cast<const long long*>(p.ocl)[s_b + key]
                                  : static_cast<long long>(static_cast<const int*>(p.ocl)[s_b + key]);
      dst = (d >= 0 && d < p.pool) ? d : -1;
      if (dst < 0 && writer && ch == 0) atomicOr(p.err, kErrBadIndex);
    }
    ksrc[key] = src;
    kdst[key] = dst;
  }
  sync();  // also publishes ksrc / kdst
  if constexpr (!CL) {
    const long long tot = (scan[0] + scan[1] + scan[2] + scan[3]) * p.n_hg;
    const long long before = scan[4] + scan[5] + scan[6] + scan[7];
    long long W = (tot + p.n_stream - 1) / p.n_stream;
    if (W < p.w_min) W = p.w_min;
    const long long off = before * p.n_hg + static_cast<long long>(sg.hg) * sg.len;
    const long long c_first = off / W, c_last = (off + sg.len - 1) / W;
    npc = c_last - c_first + 1;  // pieces of the segment
    slot0 = c_first + s_idx;     // partial of piece i, this head: (slot0 + i) HC + hc
  }

  // Everything above reads only the call's inputs.  The combine kernel is
  // launched as a programmatic dependent of the stream launch, so it may have
  // started while the stream still runs: wait for that grid to complete (and
  // its partials to be visible) before reading them.  Without such a launch
  // the wait returns at once.
  if constexpr (!CL) asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- stage the pieces: batch k (pieces k nb .. k nb + nb - 1) into half k % 2 ----
  // Thread t copies (and later folds) row t / 8, 16-byte chunk t % 8 of every
  // piece's 16 x 32 block; lane u < n of each warp copies piece u's four
  // log-sum-exps of the warp's rows.  One cp.async group per batch.  The
  // cluster form's pieces (at most 2 nb: its CTAs) go in one batch.
  const int nb = max(1, min(p.cmb_nb, kBatchMax));  // the host's choice, within what the copies serve
  if (CL && npc > 2 * nb) {
    // the host sizes the cluster form's slots for its cluster: never taken
    if (flagger) atomicOr(p.err, kErrBadKvIndptr);
    npc = 2 * nb;
  }
  const long long nbatch = CL ? 1 : (npc + nb - 1) / nb;
  unsigned char* blk = smem + kStageOff;
  unsigned char* lse_st = blk + 2 * nb * kPieceBytes;
  const int fr = tid >> 3, fch = tid & 7;  // row of the tile, 16-byte chunk of the 32 columns
  auto batch_n = [&](long long k) -> int {
    return CL ? static_cast<int>(npc) : static_cast<int>(min(static_cast<long long>(nb), npc - k * nb));
  };
  auto batch_h0 = [&](long long k) -> int { return CL ? 0 : static_cast<int>(k & 1) * nb; };
  auto issue = [&](long long k) {
    const long long i0 = k * nb;
    const int n = batch_n(k);
    const int h0 = batch_h0(k);
    for (int u = 0; u < n; ++u) {
      const long long sl = (slot0 + i0 + u) * p.HC + hc;
      cp_async_16(smem_u32(blk + (h0 + u) * kPieceBytes + fr * (kCols * 4) + fch * 16),
                  p.po + (sl * RM + 16 * tile + fr) * D + col0 + fch * 4);
    }
    if (lane < n) {
      const long long sl = (slot0 + i0 + lane) * p.HC + hc;
      cp_async_16(smem_u32(lse_st + (h0 + lane) * kPieceLseBytes + warp * 16), p.plse + sl * RM + 16 * tile + 4 * warp);
    }
    cp_async_commit();
  };
  issue(0);
  if (nbatch > 1) issue(1);

  // ---- stage the draft K rows (whole head dimension) and this slice of V ----
  // Plain drafts (k_extend / v_extend, no store) go by cp.async, one group
  // committed after the first two batches, and land while the pieces are
  // folded; the cache and store forms convert in registers.
  const int LK = (p.L + 7) & ~7;  // whole 8-key groups (keys past L staged as zero)
  unsigned char* kst = smem + kKOff;
  unsigned char* vst = smem + kVOff;
  const bool plain_drafts = !p.paged && p.wmode == 0;
  if (plain_drafts) {
    for (int idx = tid; idx < LK * (D / 2); idx += kThreads) {
      const int key = idx / (D / 2), d = (idx % (D / 2)) * 2;
      unsigned char* dk = kst + key * kKPitch + d * 2;
      if (key < p.L)
        cp_async_4(smem_u32(dk), p.ke + ksrc[key] * p.ke_s0 + static_cast<long long>(kvh) * p.ke_s1 + d);
      else
        *reinterpret_cast<uint32_t*>(dk) = 0u;
    }
    for (int idx = tid; idx < p.L * (kCols / 2); idx += kThreads) {
      const int key = idx / (kCols / 2), c = (idx % (kCols / 2)) * 2;
      cp_async_4(smem_u32(vst + (key * kCols + c) * 2),
                 p.ve + ksrc[key] * p.ve_s0 + static_cast<long long>(kvh) * p.ve_s1 + col0 + c);
    }
    cp_async_commit();
  }

  if (!plain_drafts) {
    for (int idx = tid; idx < LK * (D / 2); idx += kThreads) {
      const int key = idx / (D / 2), d = (idx % (D / 2)) * 2;
      uint32_t val = 0u;
      const long long src = key < p.L ? ksrc[key] : -1;
      if (src >= 0) {
        if (p.paged && p.wmode != 2) {
          const unsigned char* kr = p.kb + src * p.kb_s0 + static_cast<long long>(kvh) * p.kb_s1;
          if constexpr (FP8)
            val = e4m3x2_to_bf16x2(*reinterpret_cast<const unsigned short*>(kr + d));
          else
            val = *reinterpret_cast<const uint32_t*>(kr + d * 2);
        } else {
          val = ld_u32(p.ke + src * p.ke_s0 + static_cast<long long>(kvh) * p.ke_s1 + d);
          const long long dst = kdst[key];
          const bool mine = writer && dst >= 0 && d >= col0 && d < col0 + kCols;
          if (p.wmode != 0) {
            const float2 x = unpack_bf16(val);
            unsigned char* kd = p.kw + (dst >= 0 ? dst : 0) * p.kb_s0 + static_cast<long long>(kvh) * p.kb_s1;
            if constexpr (FP8) {
              const unsigned short c = store_e4m3x2(x.x, x.y, p.kq);
              if (mine) *reinterpret_cast<unsigned short*>(kd + d) = c;
              if (p.wmode == 2) val = e4m3x2_to_bf16x2(c);  // attend over the stored values
            } else {
              const uint32_t c = store_bf16x2(x.x, x.y, p.kq);
              if (mine) *reinterpret_cast<uint32_t*>(kd + d * 2) = c;
              if (p.wmode == 2) val = c;
            }
          }
        }
      }
      *reinterpret_cast<uint32_t*>(kst + key * kKPitch + d * 2) = val;
    }
    for (int idx = tid; idx < p.L * (kCols / 2); idx += kThreads) {
      const int key = idx / (kCols / 2), c = col0 + (idx % (kCols / 2)) * 2;
      uint32_t val = 0u;  // bf16 x2 (every staged value is a bf16 value)
      const long long src = ksrc[key];
      if (src >= 0) {
        if (p.paged && p.wmode != 2) {
          const unsigned char* vr = p.vb + src * p.vb_s0 + static_cast<long long>(kvh) * p.vb_s1;
          if constexpr (FP8)
            val = e4m3x2_to_bf16x2(*reinterpret_cast<const unsigned short*>(vr + c));
          else
            val = *reinterpret_cast<const uint32_t*>(vr + c * 2);
        } else {
          val = ld_u32(p.ve + src * p.ve_s0 + static_cast<long long>(kvh) * p.ve_s1 + c);
          const long long dst = kdst[key];
          if (p.wmode != 0) {
            const float2 v = unpack_bf16(val);
            unsigned char* vd = p.vw + (dst >= 0 ? dst : 0) * p.vb_s0 + static_cast<long long>(kvh) * p.vb_s1;
            const bool mine = writer && dst >= 0;
            if constexpr (FP8) {
              const unsigned short cv = store_e4m3x2(v.x, v.y, p.vq);
              if (mine) *reinterpret_cast<unsigned short*>(vd + c) = cv;
              if (p.wmode == 2) val = e4m3x2_to_bf16x2(cv);
            } else {
              const uint32_t cv = store_bf16x2(v.x, v.y, p.vq);
              if (mine) *reinterpret_cast<uint32_t*>(vd + c * 2) = cv;
              if (p.wmode == 2) val = cv;
            }
          }
        }
      }
      *reinterpret_cast<uint32_t*>(vst + (key * kCols + (c - col0)) * 2) = val;
    }
  }

  // ---- this warp's query fragments: rows of the tile, head dims [DW warp, DW warp + DW) ----
  uint32_t qf[KSW][4];
  {
    const int r0 = 16 * tile + g;
    load_q<KSW>(p, sg, hc, r0, r0 + 8, j, false, qf, DW * warp);
  }

  // ---- fold: this thread's row and four columns over every piece, in piece order ----
  float fm = NEG_INF, fl = 0.f, fa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (long long k = 0; k < nbatch; ++k) {
    // groups committed after batch k: batch k + 1 (if any) and, for k < 2,
    // the plain drafts' group (committed after batch 1)
    cp_async_wait_dyn((k + 1 < nbatch ? 1 : 0) + (k < 2 && plain_drafts ? 1 : 0));
    __syncwarp();  // the warp's log-sum-exp copies
    const int n = batch_n(k);
    const int h0 = batch_h0(k);
#pragma unroll 1
    for (int u = 0; u < n; ++u) {
      const float x = *reinterpret_cast<const float*>(lse_st + (h0 + u) * kPieceLseBytes + fr * 4);
      if (x == NEG_INF) continue;  // a piece with nothing visible
      const float4 v = *reinterpret_cast<const float4*>(blk + (h0 + u) * kPieceBytes + fr * (kCols * 4) + fch * 16);
      if (x > fm) {
        const float sc = exp2f(fm - x);  // 0 while fm is -inf
        fa[0] *= sc;
        fa[1] *= sc;
        fa[2] *= sc;
        fa[3] *= sc;
        fl *= sc;
        fm = x;
      }
      const float w = exp2f(x - fm);
      fa[0] = fmaf(w, v.x, fa[0]);
      fa[1] = fmaf(w, v.y, fa[1]);
      fa[2] = fmaf(w, v.z, fa[2]);
      fa[3] = fmaf(w, v.w, fa[3]);
      fl += w;
    }
    if constexpr (!CL) {
      __syncwarp();  // every lane is done with half k % 2 before it is refilled
      if (k + 2 < nbatch) issue(k + 2);
    }
  }
  cp_async_wait<0>();
  sync();  // staged drafts

  // ---- draft scores: this warp's DW-wide part of q . k for every 8-key group ----
  float* scp = reinterpret_cast<float*>(smem + kScOff) + warp * 16 * kScPitch;
#pragma unroll 1
  for (int nt = 0; nt * 8 < p.L; ++nt) {
    float sd[4] = {0.f, 0.f, 0.f, 0.f};
    const unsigned char* kr = kst + (nt * 8 + g) * kKPitch + (DW * warp) * 2;
#pragma unroll
    for (int kk = 0; kk < KSW; ++kk) {
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr + (kk * 16 + 2 * j) * 2);
      const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + (kk * 16 + 8 + 2 * j) * 2);
      mma_bf16(sd, qf[kk], b0, b1);
    }
    scp[g * kScPitch + nt * 8 + 2 * j] = sd[0];
    scp[g * kScPitch + nt * 8 + 2 * j + 1] = sd[1];
    scp[(g + 8) * kScPitch + nt * 8 + 2 * j] = sd[2];
    scp[(g + 8) * kScPitch + nt * 8 + 2 * j + 1] = sd[3];
  }
  sync();

  // ---- per thread: row r of the tile, 4 output columns (the fold's own) ----
  const int r = fr, c4 = fch * 4;
  const int prow = 16 * tile + r;
  const float M = fm;
  float acc[4] = {fa[0], fa[1], fa[2], fa[3]};
  float l = fl;
  // draft visibility: causal, or the tree mask rows (row-major [L][P+L], only
  // the draft columns are read; inconsistent offsets fall back to causal)
  long long mbase = -1;
  if (p.cmask) {
    const long long m0 = p.mindptr64 ? static_cast<const long long*>(p.mindptr)[sg.b]
                                     : static_cast<long long>(static_cast<const int*>(p.mindptr)[sg.b]);
    const long long span = static_cast<long long>(p.L) * (sg.P + p.L);
    if (m0 >= 0 && m0 + span <= p.n_mask)
      mbase = m0;
    else if (flagger)
      atomicOr(p.err, kErrBadMaskIndptr);
  }
  const int irow = prow / p.gq;  // draft index of the row
  const float* sc_all = reinterpret_cast<const float*>(smem + kScOff);
  auto score = [&](int key) -> float {
    if (key >= p.L || irow >= p.L || ksrc[key] < 0) return NEG_INF;
    const bool vis = mbase < 0 ? key <= irow
                               : __ldg(p.cmask + mbase + static_cast<long long>(irow) * (sg.P + p.L) + sg.P + key) != 0;
    if (!vis) return NEG_INF;
    float x = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) x += sc_all[(w * 16 + r) * kScPitch + key];
    return x * p.dscale2;
  };
  float mx = M;
#pragma unroll 1
  for (int key = 0; key < p.L; ++key) mx = fmaxf(mx, score(key));
  const float ms = (mx == NEG_INF) ? 0.f : mx;
  const float a = exp2f(M - ms);  // 0 when no piece had a visible key
  l *= a;
#pragma unroll
  for (int c = 0; c < 4; ++c) acc[c] *= a;
#pragma unroll 1
  for (int key = 0; key < p.L; ++key) {
    const float pk = exp2f(score(key) - ms);
    if (pk == 0.f) continue;
    l += pk;
    const float wv = pk * p.dvs;
    const uint2 vv = *reinterpret_cast<const uint2*>(vst + (key * kCols + c4) * 2);
    const float2 v0 = unpack_bf16(vv.x), v1 = unpack_bf16(vv.y);
    acc[0] = fmaf(wv, v0.x, acc[0]);
    acc[1] = fmaf(wv, v0.y, acc[1]);
    acc[2] = fmaf(wv, v1.x, acc[2]);
    acc[3] = fmaf(wv, v1.y, acc[3]);
  }
  // a row with nothing visible (empty prefix, no visible draft) is 0
  if (prow < p.R) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16* op = p.o + (static_cast<long long>(s_b) + prow / p.gq) * p.o_s0 +
                        static_cast<long long>(kvh * p.gq + prow % p.gq) * p.o_s1 + col0 + c4;
    *reinterpret_cast<uint32_t*>(op) = pack_bf16(acc[0] * inv, acc[1] * inv);
    *reinterpret_cast<uint32_t*>(op + 2) = pack_bf16(acc[2] * inv, acc[3] * inv);
  }
}

template <int D, bool FP8>
__global__ void __launch_bounds__(cmb::kThreads) vsk_combine_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int kSlices = cmb::Geo<D>::kSlices;
  const int ch = static_cast<int>(blockIdx.x % kSlices);
  const int tile = static_cast<int>((blockIdx.x / kSlices) % p.MT);
  const int hc = static_cast<int>((blockIdx.x / (kSlices * p.MT)) % p.HC);
  const long long s_idx = static_cast<long long>(blockIdx.x) / (kSlices * p.MT * p.HC);
  combine_unit<D, FP8, false>(p, smem, static_cast<int>(threadIdx.x), 0, s_idx, hc, tile, ch, 0, 0);
}
