// sv_chain.cuh -- chain verification (one chain of K drafts per request).
//
// The step follows Algorithm 1 as restated in the CMU 15-779 Lecture 17
// notes ("Speculative Decoding", sec. 2.4) and the study notes "LLM
// speculative decoding 02" (sec. 4): accept draft x_i iff
// u_i * q_i(x_i) < p_i(x_i), stop at the first rejection n, emit a draw
// from norm(max(0, p_n - q_n)) -- or, if all drafts pass, from p_{nd} --
// by inverse CDF with u_K.  Greedy requests (t == 0) accept iff x_i is the
// argmax of target row i (lecture notes sec. 2.2; study notes sec. 10).
//
// Inside the persistent kernel (sv_kernel.cuh):
//   main pass   every row the step reads is reduced chunk by chunk to
//               (max, sum exp) or (max, lowest argmax), one 64-bit partial
//               per chunk, on the streaming CTAs;
//   request     a warp of a control CTA polls the request's partials as
//   finalize    they are written, merges its rows, runs the accept tests
//               and the prefix-terminating scan; a greedy request is then
//               complete, a sampled one publishes its draw (row pair n) as
//               a self-marking record, then writes the accepted prefix;
//   draw pass   the streaming CTAs' scouts, each walking its static share
//               of the draw claims, stream the published row pairs again
//               as draw chunks (16 KB of p_n | 16 KB of q_n); each consumer
//               warp turns its 256-token segments into residual weights and
//               their sums;
//   draw        the same control warp polls the draw's segment sums, takes
//   finalize    the float-pair prefix over them, finds the segment holding
//               u * S, rescans it with bit-identical arithmetic and writes
//               the emitted token.
#pragma once

#include "sv_kernel.cuh"

namespace sv {

struct ChainProblem {
  static constexpr int kAuxBytes = 0;
  static constexpr bool kWarpFinalize = true;
  static constexpr bool kHasDraws = true;
  static constexpr bool kHasDirectFin = true;  // top-k requests: finalize only
  static constexpr bool kCtrl = true;          // finalizes run on control CTAs
  int n_req, K, V, es, ipr, chunk_el, max_topk;
  int n_ctrl;        // control CTAs (the last n_ctrl of the grid); they stream nothing
  int ipr2, chunk2;  // draw pass: chunks per row pair, tokens per chunk
  bool bulk;
  const char* target;
  int64_t t_stride;  // bytes between target rows
  const char* draft;
  int64_t d_stride;
  const int* tokens;
  const int* num_drafts;
  const float* temperature;
  const int* top_k;
  const float* uniforms;
  int* out_tokens;
  int* out_len;
  int* accept_len;
  float* p_at;
  float* q_at;
  unsigned long long* jobs;  // [SV_MAX_B][kJobWords] the draw of request b (see P2Job)
  const float2* topk_lists;  // [B (2K+1)][max_topk] top-k (logit, id) of row (b, i), token order
  const float2* topk_mz;     // [B (2K+1)] (m, Z) over those logits
  Ws ws;

  __device__ void write_failed(int b, int flag) const {
    for (int i = 0; i <= K; ++i) out_tokens[static_cast<size_t>(b) * (K + 1) + i] = -1;
    out_len[b] = 0;
    accept_len[b] = 0;
    if (p_at)
      for (int i = 0; i < K; ++i) p_at[static_cast<size_t>(b) * K + i] = __int_as_float(0x7fc00000);
    if (q_at)
      for (int i = 0; i < K; ++i) q_at[static_cast<size_t>(b) * K + i] = __int_as_float(0x7fc00000);
    record_error(&ws.hdr->error, flag);
  }

  // Before the launch may read its inputs (the wait on the preceding work):
  // ask L2 for the lines of the per-request arguments the preamble reads.
  // A prefetch is only a hint and L2 is the point of coherence, so it can
  // return no stale value.
  __device__ void prefetch_args(int lane) const {
    if (32 * lane >= n_req) return;
    prefetch_l2(temperature + 32 * lane);
    if (num_drafts) prefetch_l2(num_drafts + 32 * lane);
    if (top_k) prefetch_l2(top_k + 32 * lane);
  }

  // Processing order: sampled requests first (their draw pass should overlap
  // the rest of the main pass), then greedy ones, each in request order.
  // rows: greedy nd+1, sampled 2nd+1; top-k requests read no rows here (the
  // top-k pass has reduced them to lists) and go straight to their
  // finalize.  Warp 0 alone: lane l takes a contiguous block of requests,
  // classifies them in one load pass (its classification goes to
  // `scratch`, the chunk ring, idle until the preamble ends), a warp scan
  // places the blocks, and a second pass over the scratch fills the
  // position tables.  The other warps go straight to the barrier after it.
  __device__ void preamble(Shared& sh, PosTables& tab, int4*, unsigned char* scratch) const {
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    int4* req = reinterpret_cast<int4*>(scratch);  // per request: kind, nd, bits of t
    const int per = (n_req + 31) / 32;
    const int lo = min(lane * per, n_req);
    const int hi = min(lo + per, n_req);
    int4 cnt = make_int4(0, 0, 0, 0);  // sampled n, sampled rows, other n, other rows
#pragma unroll 4
    for (int b = lo; b < hi; ++b) {
      const int nd = num_drafts ? num_drafts[b] : K;
      const float t = temperature[b];
      const int kind = chain_kind(nd, t, top_k ? top_k[b] : 0, K, V, max_topk, draft != nullptr);
      req[b] = make_int4(kind, nd, __float_as_int(t), 0);
      const int rows = kind < 0 ? 0 : (kind == KIND_ARGMAX ? nd + 1 : (kind == KIND_TOPK ? 0 : 2 * nd + 1));
      if (kind == KIND_SOFTMAX) {
        cnt.x += 1;
        cnt.y += rows;
      } else {
        cnt.z += 1;
        cnt.w += rows;
      }
    }
    int4 inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int4 y = make_int4(__shfl_up_sync(0xffffffffu, inc.x, o), __shfl_up_sync(0xffffffffu, inc.y, o),
                               __shfl_up_sync(0xffffffffu, inc.z, o), __shfl_up_sync(0xffffffffu, inc.w, o));
      if (lane >= o) {
        inc.x += y.x;
        inc.y += y.y;
        inc.z += y.z;
        inc.w += y.w;
      }
    }
    const int4 tot = make_int4(__shfl_sync(0xffffffffu, inc.x, 31), __shfl_sync(0xffffffffu, inc.y, 31),
                               __shfl_sync(0xffffffffu, inc.z, 31), __shfl_sync(0xffffffffu, inc.w, 31));
    int hpos = inc.x - cnt.x, hrow = inc.y - cnt.y;
    int lpos = tot.x + inc.z - cnt.z, lrow = tot.y + inc.w - cnt.w;
    for (int b = lo; b < hi; ++b) {
      const int4 r = req[b];
      const int kind = r.x, nd = r.y;
      int pos, rows = 0;
      if (kind == KIND_SOFTMAX) {
        rows = 2 * nd + 1;
        pos = hpos++;
        tab.rstart[pos] = hrow;
        hrow += rows;
      } else {
        rows = kind == KIND_ARGMAX ? nd + 1 : 0;
        pos = lpos++;
        tab.rstart[pos] = lrow;
        lrow += rows;
      }
      tab.info[pos] = make_info(b, kind < 0 ? 0 : kind, nd < 0 ? 0 : min(nd, 0x7ff));
      const Scale2 c = scale_for(__int_as_float(r.z));
      tab.scale[pos] = make_float2(c.hi, c.lo);
      if (kind < 0 && blockIdx.x == 0) write_failed(b, 0x20);
    }
    if (lane == 0) {
      tab.rstart[n_req] = tot.y + tot.w;
      sh.n_pos = n_req;
      sh.n_draw_cap = tot.x;
    }
  }

  __device__ const char* trow(int b, int i) const {
    return target + (static_cast<int64_t>(b) * (K + 1) + i) * t_stride;
  }
  __device__ const char* drow(int b, int i) const {
    return draft + (static_cast<int64_t>(b) * K + i) * d_stride;
  }

  __device__ void fill_stage(const PosTables& tab, int rl, StageMeta& mt, ResMeta& rm) const {
    const int info = tab.info[mt.pos];
    const int b = info_req(info), nd = info_extra(info);
    mt.kind = info_kind(info);
    const float2 s = tab.scale[mt.pos];
    mt.c_hi = s.x;
    mt.c_lo = s.y;
    const char* rp = rl <= nd ? trow(b, rl) : drow(b, rl - nd - 1);
    mt.src = rp + static_cast<size_t>(mt.el_base) * es;
    rm.tkt = b;
    rm.need = (tab.rstart[mt.pos + 1] - tab.rstart[mt.pos]) * ipr;
    rm.fin_code = mt.pos;
  }

  // Publish request b's draw (or its failure) as three self-marking words.
  __device__ void publish_job(int b, const P2Job* jb) const {
    unsigned long long* w = jobs + static_cast<size_t>(b) * kJobWords;
    if (jb) {
      st_relaxed_u64(w, __float_as_uint(jb->izp) |
                            static_cast<unsigned long long>(__float_as_uint(jb->mp)) << 32);
      const unsigned lo = jb->mode == 0 ? __float_as_uint(jb->izq) : 0x80000000u;
      st_relaxed_u64(w + 1, lo | static_cast<unsigned long long>(__float_as_uint(jb->mq)) << 32);
      st_relaxed_u64(w + 2, static_cast<unsigned long long>(1 + jb->n + (jb->mode << 8)));
    } else {
      st_relaxed_u64(w, 0x80000000ull);
      st_relaxed_u64(w + 1, 0x80000000ull);
      st_relaxed_u64(w + 2, 1ull | 1ull << 32);
    }
  }
  // Decode the words of request b's draw (all nonzero); false if it failed.
  __device__ bool decode_job(int b, const unsigned long long (&w)[3], Scale2 c, P2Job& j) const {
    const unsigned meta = static_cast<unsigned>(w[2]);
    j.b = b;
    j.n = static_cast<int>(meta & 0xffu) - 1;
    j.mode = static_cast<int>(meta >> 8);
    j.izp = __uint_as_float(static_cast<unsigned>(w[0]));
    j.mp = __uint_as_float(static_cast<unsigned>(w[0] >> 32));
    j.izq = j.mode == 0 ? __uint_as_float(static_cast<unsigned>(w[1])) : 0.f;
    j.mq = __uint_as_float(static_cast<unsigned>(w[1] >> 32));
    j.c_hi = c.hi;
    j.c_lo = c.lo;
    return (w[2] >> 32) == 0ull;
  }
  // The draw at position d of the processing order (sampled requests hold
  // positions 0 .. number of sampled requests - 1), polled until published:
  // returns 1 (a draw), 0 (the request failed: no draw) or -1 (the wait
  // expired).
  __device__ int poll_job(const PosTables& tab, int d, uint64_t limit, P2Job& j) const {
    const int b = info_req(tab.info[d]);
    const unsigned long long* p = jobs + static_cast<size_t>(b) * kJobWords;
    unsigned long long w[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) w[k] = ld_relaxed_u64(p + k);
    const uint64_t t0 = globaltimer_ns();
    unsigned backoff = 32;
    while (w[0] == 0ull || w[1] == 0ull || w[2] == 0ull) {
      if (globaltimer_ns() - t0 > limit) return -1;
      __nanosleep(backoff);
      backoff = min(backoff * 2u, 128u);
#pragma unroll
      for (int k = 0; k < 3; ++k)
        if (w[k] == 0ull) w[k] = ld_relaxed_u64(p + k);
    }
    j.pos = d;
    return decode_job(b, w, Scale2{tab.scale[d].x, tab.scale[d].y}, j) ? 1 : 0;
  }
  // The draw of the request at position pos, read back by the warp that
  // published it.
  __device__ P2Job load_job(const PosTables& tab, int pos) const {
    const int b = info_req(tab.info[pos]);
    const unsigned long long* p = jobs + static_cast<size_t>(b) * kJobWords;
    unsigned long long w[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) w[k] = ld_relaxed_u64(p + k);
    P2Job j;
    j.pos = pos;
    decode_job(b, w, Scale2{tab.scale[pos].x, tab.scale[pos].y}, j);
    return j;
  }

  // segments of kRSeg tokens per draw chunk; a consumer warp takes
  // segs_per_chunk / kGroupWarps of them (kSpwBf16 or kSpwF32)
  __device__ int segs_per_chunk() const { return chunk2 / kRSeg; }

  __device__ void fill_resid(const P2Job& jb, int chunk, StageMeta& mt, ResMeta& rm) const {
    mt.kind = KIND_RESID_PASS;
    mt.el_base = chunk * chunk2;
    mt.n_el = min(chunk2, V - mt.el_base);
    mt.c_hi = jb.c_hi;
    mt.c_lo = jb.c_lo;
    mt.aux = make_float4(jb.mp, jb.izp, jb.mq, jb.izq);
    mt.sub = jb.mode;
    mt.src = trow(jb.b, jb.n) + static_cast<size_t>(mt.el_base) * es;
    mt.src2 = jb.mode == 0 ? drow(jb.b, jb.n) + static_cast<size_t>(mt.el_base) * es : nullptr;
    rm.slot = (jb.b * ipr2 + chunk) * segs_per_chunk();
    rm.tkt = kDrawTicketBase + jb.b;
    rm.need = ipr2;
    rm.fin_code = jb.pos | kFinResid;
  }

  // draw pass: warp w of the group reduces segments w * spw + s (s < spw)
  // of the chunk, lane l tokens [8 l, 8 l + 8) of each; returns the
  // segment sums.  Staged data is held packed until the stage is released.
  __device__ float4 consume_resid(const StageMeta& mt, const unsigned char* sp,
                                  uint64_t* empty_bar, int ctid, int lane) const {
    const int warp = ctid >> 5;
    const int spw = segs_per_chunk() / kGroupWarps;  // kSpwBf16 or kSpwF32
    const int mode = mt.sub;
    const ResidParams r{mt.aux.x, mt.aux.y, mt.aux.z, mt.aux.w, Scale2{mt.c_hi, mt.c_lo}, mode};
    float tot[4] = {0.f, 0.f, 0.f, 0.f};
    auto seg_sum = [&](const float* xp, const float* xq, int t0) {
      float w[8];
      const float ls = resid_weights8(xp, xq, t0, mt.n_el, r, w);
      return __shfl_sync(0xffffffffu, warp_incl_scan_rn(ls, lane), 31);
    };
    const char* pb = reinterpret_cast<const char*>(sp);
    const char* qb = pb + kChunkBytes / 2;
    if (bulk && es == 2) {
      uint4 pv[kSpwBf16], qv[kSpwBf16];
#pragma unroll
      for (int s = 0; s < kSpwBf16; ++s) {
        const int t0 = (warp * kSpwBf16 + s) * kRSeg + lane * 8;
        pv[s] = *reinterpret_cast<const uint4*>(pb + t0 * 2);
        qv[s] = mode == 0 ? *reinterpret_cast<const uint4*>(qb + t0 * 2) : make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
#pragma unroll
      for (int s = 0; s < kSpwBf16; ++s) {
        const int t0 = (warp * kSpwBf16 + s) * kRSeg + lane * 8;
        float xp[8], xq[8];
        const uint32_t wp[4] = {pv[s].x, pv[s].y, pv[s].z, pv[s].w};
        const uint32_t wq[4] = {qv[s].x, qv[s].y, qv[s].z, qv[s].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          xp[2 * h] = bf16lo(wp[h]);
          xp[2 * h + 1] = bf16hi(wp[h]);
          xq[2 * h] = mode == 0 ? bf16lo(wq[h]) : kNegInf;
          xq[2 * h + 1] = mode == 0 ? bf16hi(wq[h]) : kNegInf;
        }
        tot[s] = seg_sum(xp, xq, t0);
      }
    } else {
      return consume_resid_cold(mt, sp, empty_bar, ctid, lane);
    }
    return make_float4(tot[0], tot[1], tot[2], tot[3]);
  }

  // The draw pass for fp32 logits or rows that were not staged: out of line,
  // so the streaming loop's code stays compact.
  __device__ __forceinline__ float4 consume_resid_cold(const StageMeta& mt, const unsigned char* sp,
                                                    uint64_t* empty_bar, int ctid, int lane) const {
    const int warp = ctid >> 5;
    const int spw = segs_per_chunk() / kGroupWarps;  // kSpwF32 (fp32) or kSpwBf16
    const int mode = mt.sub;
    const ResidParams r{mt.aux.x, mt.aux.y, mt.aux.z, mt.aux.w, Scale2{mt.c_hi, mt.c_lo}, mode};
    float tot[4] = {0.f, 0.f, 0.f, 0.f};
    auto seg_sum = [&](const float* xp, const float* xq, int t0) {
      float w[8];
      const float ls = resid_weights8(xp, xq, t0, mt.n_el, r, w);
      return __shfl_sync(0xffffffffu, warp_incl_scan_rn(ls, lane), 31);
    };
    const char* pb = reinterpret_cast<const char*>(sp);
    const char* qb = pb + kChunkBytes / 2;
    if (bulk) {
      float4 pv[kSpwF32][2], qv[kSpwF32][2];
#pragma unroll
      for (int s = 0; s < kSpwF32; ++s) {
        const int t0 = (warp * kSpwF32 + s) * kRSeg + lane * 8;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          pv[s][h] = *reinterpret_cast<const float4*>(pb + t0 * 4 + 16 * h);
          qv[s][h] = mode == 0 ? *reinterpret_cast<const float4*>(qb + t0 * 4 + 16 * h)
                               : make_float4(kNegInf, kNegInf, kNegInf, kNegInf);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
#pragma unroll
      for (int s = 0; s < kSpwF32; ++s) {
        const int t0 = (warp * kSpwF32 + s) * kRSeg + lane * 8;
        const float xp[8] = {pv[s][0].x, pv[s][0].y, pv[s][0].z, pv[s][0].w,
                             pv[s][1].x, pv[s][1].y, pv[s][1].z, pv[s][1].w};
        const float xq[8] = {qv[s][0].x, qv[s][0].y, qv[s][0].z, qv[s][0].w,
                             qv[s][1].x, qv[s][1].y, qv[s][1].z, qv[s][1].w};
        tot[s] = seg_sum(xp, xq, t0);
      }
    } else {
      // rows not fit for bulk copies: nothing was staged, read them here
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
      for (int s = 0; s < spw; ++s) {
        const int t0 = (warp * spw + s) * kRSeg + lane * 8;
        float xp[8], xq[8];
        load8(mt.src, es, false, t0, mt.n_el, xp);
        load8(mt.src2, es, false, t0, mode == 0 ? mt.n_el : 0, xq);
        const float v = seg_sum(xp, xq, t0);
        if (s == 0) tot[0] = v;
        else if (s == 1) tot[1] = v;
        else if (s == 2) tot[2] = v;
        else tot[3] = v;
      }
    }
    return make_float4(tot[0], tot[1], tot[2], tot[3]);
  }

  // A row chunk's partial as one 64-bit word that control CTAs poll: (max,
  // sum) for softmax rows, (max, lowest index + 1) for argmax rows.  Never
  // all zero (a sum is at least 1 unless the maximum is -inf or NaN; the
  // index word is at least 1), so zero marks a slot not yet written.
  __device__ void store_partial(int slot, int kind, float2 v) const {
    const unsigned hi = kind == KIND_ARGMAX ? static_cast<unsigned>(__float_as_int(v.y)) + 1u
                                            : __float_as_uint(v.y);
    st_relaxed_u64(reinterpret_cast<unsigned long long*>(ws.partials + slot),
                   (static_cast<unsigned long long>(hi) << 32) | __float_as_uint(v.x));
  }
  // A draw chunk's segment sums of consumer warp w (spw of them), stored
  // sign-flipped (enc_seg: never the zero word) where the draw finalize
  // polls them; zero marks a sum not yet written.
  __device__ void store_segsums_warp(int base, int w, float4 v) const {
    const int spw = segs_per_chunk() / kGroupWarps;
    unsigned* d = reinterpret_cast<unsigned*>(ws.segsums) + base + w * spw;
    const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (k < spw)
        asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(d + k), "r"(enc_seg(x[k]))
                     : "memory");
  }
  __device__ void store_segsums(const ResMeta& rm, int lane, float4 v) const {
    if (lane < kGroupWarps) store_segsums_warp(rm.slot, lane, v);
  }
  __device__ float4 consume(const StageMeta& mt, const unsigned char* sp, uint64_t* empty_bar,
                            int ctid, int lane) const {
    if (mt.kind == KIND_RESID_PASS) return consume_resid(mt, sp, empty_bar, ctid, lane);
    const float2 r = reduce_row_chunk(mt, sp, empty_bar, ctid, lane, bulk, es);
    return make_float4(r.x, r.y, 0.f, 0.f);
  }

  // a request whose finalize needs no main-pass rows
  __device__ bool direct_fin(const PosTables& tab, int pos) const {
    return info_kind(tab.info[pos]) == KIND_TOPK;
  }
  __device__ void finalize_warp(Shared& sh, const PosTables& tab, int code, int lane,
                                WarpFin& wf) const {
    if (code & kFinResid) draw_finalize(sh, tab, code & ~kFinResid, lane, wf);
    else if (info_kind(tab.info[code]) == KIND_TOPK) topk_finalize(tab, code, lane, wf);
    else request_finalize(sh, tab, code, lane, wf);
  }
  // Control CTAs: the finalize of position pos (returns 1 when it published
  // a draw), and the draw finalize of a published draw.  Each polls the data
  // words it needs -- the request's chunk partials, the draw's segment sums
  // -- with bounded waits: every word is written once per call and is never
  // zero once written, so no count or fence stands between the last chunk
  // and its finalize.
  __device__ int ctrl_request(Shared& sh, const PosTables& tab, int pos, int lane,
                              WarpFin& wf) const {
    const int info = tab.info[pos];
    const int kind = info_kind(info);
    const int rows = tab.rstart[pos + 1] - tab.rstart[pos];
    if (kind == KIND_TOPK) {
      topk_finalize(tab, pos, lane, wf);
      return 0;
    }
    if (rows == 0) return 0;  // invalid arguments: failed in the preamble
    const int drew = request_finalize(sh, tab, pos, lane, wf);
    // leave the request's partial slots zero for the next call
    unsigned long long* w =
        reinterpret_cast<unsigned long long*>(ws.partials) + static_cast<size_t>(tab.rstart[pos]) * ipr;
    for (int j = lane; j < rows; j += 32)
      for (int c = 0; c < ipr; ++c) st_relaxed_u64(w + static_cast<size_t>(j) * ipr + c, 0ull);
    return drew;
  }
  __device__ void ctrl_draw(Shared& sh, const PosTables& tab, int pos, int lane,
                            WarpFin& wf) const {
    draw_finalize(sh, tab, pos, lane, wf);
  }
  __device__ void topk_finalize(const PosTables& tab, int pos, int lane, WarpFin& wf) const;
  __device__ int request_finalize(Shared& sh, const PosTables& tab, int pos, int lane,
                                   WarpFin& wf) const;
  __device__ void draw_finalize(Shared& sh, const PosTables& tab, int pos, int lane,
                                WarpFin& wf) const;
  // A claim of the failed draw at position d (the record says failed): the
  // ipr2 claims of the draw each count themselves in the record's spare
  // word, and the last one clears the record for the next call -- every
  // other claim has read it by then.
  __device__ void failed_claim(const PosTables& tab, int d) const {
    unsigned long long* w = jobs + static_cast<size_t>(info_req(tab.info[d])) * kJobWords;
    if (atomicAdd(w + 3, 1ull) == static_cast<unsigned long long>(ipr2 - 1))
      for (int k = 0; k < kJobWords; ++k) st_relaxed_u64(w + k, 0ull);
  }
};

// Eight consecutive chunk partials of a row (words c0 .. c0 + 7 below n;
// `fill` for the rest), polled until every one is written: a written word
// is never zero.  The back-off is short, and shorter once part of the batch
// is in, since the rest of a row lands within a chunk time: the finalize
// that follows is on the step's critical path.  False when the wait
// expired.
__device__ __forceinline__ bool poll_words8(const unsigned long long* w, int c0, int n,
                                            unsigned long long fill, unsigned long long (&t)[8],
                                            uint64_t t0, uint64_t limit) {
#pragma unroll
  for (int k = 0; k < 8; ++k) t[k] = c0 + k < n ? ld_relaxed_u64(w + c0 + k) : fill;
  unsigned backoff = 64;
  for (;;) {
    int missing = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) missing += t[k] == 0ull;
    if (missing == 0) return true;
    if (globaltimer_ns() - t0 > limit) return false;
    __nanosleep(backoff);
    backoff = missing < 8 ? 32u : min(backoff * 2u, 256u);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (t[k] == 0ull) t[k] = ld_relaxed_u64(w + c0 + k);
  }
}

__device__ __forceinline__ float2 word_f2(unsigned long long v) {
  return make_float2(__uint_as_float(static_cast<unsigned>(v)),
                     __uint_as_float(static_cast<unsigned>(v >> 32)));
}

// Merge the chunk partials of a request's rows into wf as they are
// written: lane j takes row j (passes of 32 rows), polls its ipr partials
// eight at a time and merges them from the polled values -- one exp2 per
// partial, no shuffles, because the consumers keep the shared-memory and
// special-function pipes of the SM busy while finalizes run.  Softmax rows:
// the maximum first, then each sum rescaled once to it; argmax rows: the
// largest value, lowest index (the partial's high word is index + 1).
// False in every lane when a wait expired.
__device__ __forceinline__ bool merge_rows(const float2* partials, int r0, int nrows, int ipr,
                                           bool greedy, Scale2 c, int lane, WarpFin& wf,
                                           uint64_t limit) {
  const uint64_t t0 = globaltimer_ns();
  bool ok = true;
  for (int j = lane; j < nrows && ok; j += 32) {
    const unsigned long long* pp =
        reinterpret_cast<const unsigned long long*>(partials) + static_cast<size_t>(r0 + j) * ipr;
    unsigned long long t[8];
    if (greedy) {
      VI v{kNegInf, 0x7fffffff};
      const unsigned long long fill =
          (static_cast<unsigned long long>(0x7fffffffu) << 32) | __float_as_uint(kNegInf);
      for (int c0 = 0; c0 < ipr && ok; c0 += 8) {
        ok = poll_words8(pp, c0, ipr, fill, t, t0, limit);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float2 f = word_f2(t[k]);
          if (c0 + k < ipr) v = vi_better(v, VI{f.x, __float_as_int(f.y) - 1});
        }
      }
      wf.rm[j] = v.v;
      wf.ridx[j] = v.i;
    } else {
      const unsigned long long fill = __float_as_uint(kNegInf);
      float M = kNegInf;
      bool nan = false;
      for (int c0 = 0; c0 < ipr && ok; c0 += 8) {
        ok = poll_words8(pp, c0, ipr, fill, t, t0, limit);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float x = word_f2(t[k]).x;
          nan |= x != x;
          M = fmaxf(M, x);
        }
      }
      float sum = 0.f;
      if (ok && !nan && M != kNegInf) {
        for (int c0 = 0; c0 < ipr; c0 += 8) {
          // t holds the last batch of the maximum pass: reload (every word
          // is written by now) unless that batch is the first
          if (c0 > 0 || ipr > 8) {
#pragma unroll
            for (int k = 0; k < 8; ++k) t[k] = c0 + k < ipr ? ld_relaxed_u64(pp + c0 + k) : fill;
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float2 f = word_f2(t[k]);
            if (f.x != kNegInf) sum += f.y * fast_exp2(scaled_arg(f.x, M, c));
          }
        }
      }
      wf.rm[j] = nan ? nan_f() : M;
      wf.rz[j] = nan ? 0.f : sum;
    }
  }
  __syncwarp();
  return __all_sync(0xffffffffu, ok);
}

__device__ int ChainProblem::request_finalize(Shared& sh, const PosTables& tab, int pos,
                                               int lane, WarpFin& wf) const {
  const int info = tab.info[pos];
  const int b = info_req(info), kind = info_kind(info), nd = info_extra(info);
  const int r0 = tab.rstart[pos];
  const int nrows = tab.rstart[pos + 1] - r0;
  const Scale2 c{tab.scale[pos].x, tab.scale[pos].y};
  const bool greedy = kind == KIND_ARGMAX;

  // loads that do not depend on the main pass go out before its partials
  // are polled: the draft tokens, their uniforms and the logits they gather
  const int x = lane < nd ? tokens[static_cast<size_t>(b) * K + lane] : 0;
  const float ui = lane < nd ? uniforms[static_cast<size_t>(b) * (K + 1) + lane] : 0.f;
  const bool x_ok = x >= 0 && x < V;
  float lx = 0.f, dx = 0.f;
  if (!greedy && lane < nd && x_ok) {
    lx = load_logit(trow(b, lane), es, x);
    dx = load_logit(drow(b, lane), es, x);
  }
  if (!merge_rows(ws.partials, r0, nrows, ipr, greedy, c, lane, wf,
                  sh.timed_out ? kWaitLimitAfterTimeoutNs : kWaitLimitNs)) {
    sh.timed_out = 1;
    if (lane == 0) {
      write_failed(b, 0x10);
      if (!greedy) publish_job(b, nullptr);
    }
    __syncwarp();
    return 0;
  }

  // accept tests (lane i = draft i) and the prefix-terminating scan
  int err = 0;
  for (int j = lane; j < nrows; j += 32) {
    if (wf.rm[j] != wf.rm[j]) err |= 0x02;
    else if (wf.rm[j] == kNegInf || (!greedy && !(wf.rz[j] > 0.f))) err |= 0x04;
  }
  bool acc = false;
  float pa = __int_as_float(0x7fc00000), qa = __int_as_float(0x7fc00000);
  if (lane < nd) {
    if (!x_ok) {
      err |= 0x01;
    } else if (greedy) {
      acc = x == wf.ridx[lane];
      pa = acc ? 1.f : 0.f;
    } else {
      const int jt = lane, jd = nd + 1 + lane;
      // p(x) = np / Zp, q(x) = nq / Zq; the test u q(x) < p(x) is taken as
      // u nq Zp < np Zq (no division).  First in fp32: np and nq to about
      // 5e-7 relative, so the two sides carry less than 2e-6 of relative
      // error between them, and when they differ by more than 4e-6 the
      // fp32 decision is the fp64 one.  Closer calls, and exponents below
      // -96 (where u nq Zp could leave the normal range), are decided in
      // fp64 -- slow on this part, but the fast path takes all but a few
      // tests per million.
      float ahp, ahq;
      const float np32 = exp2_scaled_pair(lx, wf.rm[jt], c, ahp);
      const float nq32 = exp2_scaled_pair(dx, wf.rm[jd], c, ahq);
      const float lhs = ui * nq32 * wf.rz[jt], rhs = np32 * wf.rz[jd];
      // Z >= 1 (the maximum's own term), so the reciprocal needs no special cases
      if (ahp >= -96.f && ahq >= -96.f && fabsf(lhs - rhs) > 4e-6f * fmaxf(lhs, rhs)) {
        acc = lhs < rhs;
        pa = np32 * rcp_fma(wf.rz[jt]);
        qa = nq32 * rcp_fma(wf.rz[jd]);
      } else {
        const double cd = static_cast<double>(c.hi) + static_cast<double>(c.lo);
        const double np = exp2_nonpos(
            (static_cast<double>(lx) - static_cast<double>(wf.rm[jt])) * cd);
        const double nq = exp2_nonpos(
            (static_cast<double>(dx) - static_cast<double>(wf.rm[jd])) * cd);
        const double zp = static_cast<double>(wf.rz[jt]), zq = static_cast<double>(wf.rz[jd]);
        acc = static_cast<double>(ui) * nq * zp < np * zq;
        pa = static_cast<float>(np) * rcp_fma(wf.rz[jt]);
        qa = static_cast<float>(nq) * rcp_fma(wf.rz[jd]);
      }
    }
  }
  err = __reduce_or_sync(0xffffffffu, err);
  const unsigned mask = __ballot_sync(0xffffffffu, acc);
  int n = mask == 0xffffffffu ? 32 : __ffs(~mask) - 1;
  n = min(n, nd);

  // a sampled request publishes its draw first -- the draw pass is the
  // longer path -- then writes its outputs
  int drew = 0;
  if (!greedy && lane == 0) {
    if (!err) {
      // the draw from norm(max(0, p_n - q_n)) (rejection) or p_nd (bonus)
      P2Job jb;
      jb.b = b;
      jb.n = n;
      jb.mode = n < nd ? 0 : 1;
      jb.mp = wf.rm[n];
      jb.izp = rcp_fma(wf.rz[n]);  // Z >= 1
      jb.mq = n < nd ? wf.rm[nd + 1 + n] : 0.f;
      jb.izq = n < nd ? rcp_fma(wf.rz[nd + 1 + n]) : 0.f;
      jb.c_hi = c.hi;
      jb.c_lo = c.lo;
      jb.pos = pos;
      publish_job(b, &jb);
      drew = 1;
    } else {
      publish_job(b, nullptr);
    }
  }

  // outputs: the accepted prefix; greedy also the emitted token
  if (lane < nd) {
    if (p_at) p_at[static_cast<size_t>(b) * K + lane] = pa;
    if (q_at) q_at[static_cast<size_t>(b) * K + lane] = qa;
  }
  for (int i = max(lane, nd); i < K; i += 32) {
    if (p_at) p_at[static_cast<size_t>(b) * K + i] = __int_as_float(0x7fc00000);
    if (q_at) q_at[static_cast<size_t>(b) * K + i] = __int_as_float(0x7fc00000);
  }
  for (int i = lane; i <= K; i += 32) {
    int v = -1;
    if (!err) {
      if (i < n) v = x;  // i < n <= nd <= 32: lane i holds draft i
      else if (i == n && greedy) v = wf.ridx[n];
    }
    out_tokens[static_cast<size_t>(b) * (K + 1) + i] = v;
  }
  __syncwarp();  // every lane's outputs before a later draw finalize overwrites one
  if (lane == 0) {
    out_len[b] = err ? 0 : n + 1;
    accept_len[b] = err ? 0 : n;
    if (err) record_error(&ws.hdr->error, err);
  }
  // 1 when a draw was published (its draw finalize follows its draw pass)
  return __shfl_sync(0xffffffffu, drew, 0);
}

// Lane l's 16 stored segment sums of page g (segments [512 g + 16 l, +16)),
// as words; beyond nseg (a multiple of 4) the encoding of zero.
__device__ __forceinline__ void load_page_words(const unsigned* ss, int nseg, int g, int lane,
                                                unsigned* w) {
  const int i0 = g * kPageSeg + lane * 16;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 f = make_uint4(0x80000000u, 0x80000000u, 0x80000000u, 0x80000000u);
    if (i0 + 4 * q < nseg) f = ld_relaxed_v4(ss + i0 + 4 * q);
    w[4 * q] = f.x;
    w[4 * q + 1] = f.y;
    w[4 * q + 2] = f.z;
    w[4 * q + 3] = f.w;
  }
}

// The same, polled until every sum of the page is written (bounded; false
// in every lane when the wait expired), decoded into v.
__device__ __forceinline__ bool poll_page(const unsigned* ss, int nseg, int g, int lane, float* v,
                                          uint64_t limit) {
  const uint64_t t0 = globaltimer_ns();
  const int i0 = g * kPageSeg + lane * 16;
  unsigned w[16];
  load_page_words(ss, nseg, g, lane, w);
  unsigned backoff = 64;
  bool ok = true;
  for (;;) {
    int missing = 0;
#pragma unroll
    for (int k = 0; k < 16; ++k) missing += w[k] == 0u;
    if (__all_sync(0xffffffffu, missing == 0)) break;
    if (globaltimer_ns() - t0 > limit) {
      ok = false;
      break;
    }
    __nanosleep(backoff);
    backoff = min(backoff * 2u, 128u);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (w[4 * q] == 0u || w[4 * q + 1] == 0u || w[4 * q + 2] == 0u || w[4 * q + 3] == 0u) {
        const uint4 f = ld_relaxed_v4(ss + i0 + 4 * q);
        w[4 * q] = f.x;
        w[4 * q + 1] = f.y;
        w[4 * q + 2] = f.z;
        w[4 * q + 3] = f.w;
      }
  }
#pragma unroll
  for (int k = 0; k < 16; ++k) v[k] = dec_seg(w[k]);
  return ok;
}

// Lane l's 16 segment sums of page g, already written, decoded into v.
__device__ __forceinline__ void load_page(const unsigned* ss, int nseg, int g, int lane, float* v) {
  unsigned w[16];
  load_page_words(ss, nseg, g, lane, w);
#pragma unroll
  for (int k = 0; k < 16; ++k) v[k] = dec_seg(w[k]);
}

// The draw from the weights of the draw pass: S = the sum of the segment
// sums, target = u_K S, the segment whose running sum first exceeds target
// (pages of 512 segments, then the lane's block of 16, then the segment),
// then the token within it.  Running sums are float pairs; the search goes
// in ascending token order throughout, as the inverse CDF does.
__device__ void ChainProblem::draw_finalize(Shared& sh, const PosTables& tab, int pos, int lane,
                                            WarpFin& wf) const {
  const int b = info_req(tab.info[pos]);
  const P2Job jb = load_job(tab, pos);
  const int n = jb.n, mode = jb.mode;
  const int nseg = ipr2 * segs_per_chunk();
  unsigned* ss = reinterpret_cast<unsigned*>(ws.segsums) + static_cast<size_t>(b) * nseg;
  const float u = uniforms[static_cast<size_t>(b) * (K + 1) + K];
  const char* pr = trow(b, n);
  const char* qr = mode == 0 ? drow(b, n) : nullptr;
  ResidParams rp{jb.mp, jb.izp, jb.mq, jb.izq, Scale2{jb.c_hi, jb.c_lo}, mode};
  const int npages = (nseg + kPageSeg - 1) / kPageSeg;
  int token = -1;
  bool timed_out = false;
  for (int attempt = 0; attempt < 2 && token < 0 && !timed_out; ++attempt) {
    if (attempt == 1) {
      if (mode != 0) break;
      // a residual of zero mass (rounding only): draw from p_n instead --
      // recompute the segment sums with the bonus weights
      rp.mode = 1;
      qr = nullptr;
      for (int k = 0; k < nseg; ++k) {
        const int t0 = k * kRSeg + lane * 8;
        float xp[8], xq[8], w[8];
        load8(pr, es, bulk, t0, V, xp);
        load8(pr, es, bulk, t0, 0, xq);
        const float ls = resid_weights8(xp, xq, t0, V, rp, w);
        const float inc = warp_incl_scan_rn(ls, lane);
        if (lane == 31) __stcg(ss + k, enc_seg(inc));
      }
      __threadfence_block();
      __syncwarp();
    }
    // page totals (kept in the warp's scratch) and S
    float v[16];
    DF S{0.f, 0.f};
    for (int g = 0; g < npages; ++g) {
      // the first pass waits for the draw pass's sums to be written
      if (attempt == 0) {
        if (!poll_page(ss, nseg, g, lane, v,
                       sh.timed_out ? kWaitLimitAfterTimeoutNs : kWaitLimitNs)) {
          sh.timed_out = 1;
          timed_out = true;
          break;
        }
      } else {
        load_page(ss, nseg, g, lane, v);
      }
      DF bs{0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 16; ++j) bs = df_add(bs, v[j]);
      const DF tot = df_shfl(warp_incl_scan_df(bs, lane), 31);
      if (lane == 0) {
        wf.rz[2 * g] = tot.hi;
        wf.rz[2 * g + 1] = tot.lo;
      }
      S = df_add(S, tot);
    }
    __syncwarp();
    if (timed_out) break;
    if (!(S.hi > 0.f)) continue;
    const DF target = df_mul(u, S);
    // the page holding target (target < S, so there is one)
    int pg = -1;
    DF base{0.f, 0.f}, run{0.f, 0.f};
    for (int g = 0; g < npages; ++g) {
      const DF nxt = df_add(run, DF{wf.rz[2 * g], wf.rz[2 * g + 1]});
      if (pg < 0 && df_lt(target, nxt)) {
        pg = g;
        base = run;
      }
      run = nxt;
    }
    if (pg < 0) continue;
    if (pg != npages - 1) load_page(ss, nseg, pg, lane, v);
    // the lane whose block holds target
    DF bs{0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 16; ++j) bs = df_add(bs, v[j]);
    const DF incl = warp_incl_scan_df(bs, lane);
    const unsigned hit = __ballot_sync(0xffffffffu, df_lt(target, df_add(base, incl)));
    if (!hit) continue;
    const int owner = __ffs(hit) - 1;
    const DF prev = df_shfl(incl, owner > 0 ? owner - 1 : 0);
    const DF lane_base = owner > 0 ? df_add(base, prev) : base;
    // the segment within the owner's block
    int k = -1;
    DF seg_base = lane_base;
    if (lane == owner) {
      DF r = lane_base;
      int lastp = -1;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const DF nx = df_add(r, v[j]);
        if (k < 0 && df_lt(target, nx)) {
          k = j;
          seg_base = r;
        }
        if (v[j] > 0.f) lastp = j;
        r = nx;
      }
      if (k < 0) {
        k = lastp;  // rounding: the last segment of the block with mass
        seg_base.hi = -1.f;
      }
      if (k >= 0) k += pg * kPageSeg + owner * 16;
    }
    k = __shfl_sync(0xffffffffu, k, owner);
    seg_base = df_shfl(seg_base, owner);
    if (k < 0) continue;
    const bool in_seg = seg_base.hi >= 0.f;
    // rescan segment k exactly as the draw pass computed it
    const int t0 = k * kRSeg + lane * 8;
    float xp[8], xq[8], w[8];
    load8(pr, es, bulk, t0, V, xp);
    load8(qr, es, bulk, t0, qr ? V : 0, xq);
    const float ls = resid_weights8(xp, xq, t0, V, rp, w);
    const float inc = warp_incl_scan_rn(ls, lane);
    float exl = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) exl = 0.f;
    int tok = -1, src;
    int lastp = -1;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (w[j] > 0.f) lastp = j;
    if (in_seg) {
      const unsigned lh = __ballot_sync(0xffffffffu, df_lt(target, df_add(seg_base, inc)));
      src = lh ? __ffs(lh) - 1 : 31;
      DF cc = df_add(seg_base, exl);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cc = df_add(cc, w[j]);
        if (tok < 0 && df_lt(target, cc)) tok = j;
      }
      if (tok < 0) tok = lastp;
      if (!lh) {
        // rounding left target beyond the segment: its last positive weight
        const unsigned lp = __ballot_sync(0xffffffffu, lastp >= 0);
        src = lp ? 31 - __clz(lp) : 31;
        tok = lastp;
      }
    } else {
      const unsigned lp = __ballot_sync(0xffffffffu, lastp >= 0);
      src = lp ? 31 - __clz(lp) : 0;
      tok = lastp;
    }
    tok = __shfl_sync(0xffffffffu, tok, src);
    token = tok < 0 ? -1 : k * kRSeg + src * 8 + tok;
  }
  if (lane == 0) {
    if (token >= 0) {
      out_tokens[static_cast<size_t>(b) * (K + 1) + n] = token;
    } else {
      for (int i = 0; i <= K; ++i) out_tokens[static_cast<size_t>(b) * (K + 1) + i] = -1;
      out_len[b] = 0;
      accept_len[b] = 0;
      record_error(&ws.hdr->error, timed_out ? 0x10 : 0x04);
    }
  }
  __syncwarp();
  // leave the segment sums and the draw's record zero: any part of the
  // workspace may serve another call's chunk partials, which must start at
  // zero, and every claim of this draw has read the record (its chunks are
  // all in)
  for (int k = lane; k < nseg; k += 32) ss[k] = 0u;
  if (lane < 3) jobs[static_cast<size_t>(b) * kJobWords + lane] = 0ull;
  __syncwarp();
}

// Finalize of a top-k request from the top-k pass's lists: row (b, i) holds
// the k largest logits of that row with their ids, in token order, and
// (m, Z) over them.  p_i(x) = exp((l - m)/t) / Z for x in p_i's list and 0
// otherwise (likewise q_i), so the accept tests look the drafts up in the
// lists; the residual max(0, p_n - q_n), or p_nd for the bonus, is nonzero
// only on p_n's list, which is already in token order for the inverse CDF.
__device__ void ChainProblem::topk_finalize(const PosTables& tab, int pos, int lane,
                                            WarpFin& wf) const {
  const int info = tab.info[pos];
  const int b = info_req(info), nd = info_extra(info);
  const int r0 = b * (2 * K + 1);   // rows (b, 0 .. 2K): target 0..nd, draft nd+1 ..
  const int nrows = 2 * nd + 1;
  const Scale2 c{tab.scale[pos].x, tab.scale[pos].y};
  const int k = top_k[b];
  auto list_of = [&](int row) { return topk_lists + static_cast<size_t>(r0 + row) * max_topk; };

  const int x = lane < nd ? tokens[static_cast<size_t>(b) * K + lane] : 0;
  const float ui = lane < nd ? uniforms[static_cast<size_t>(b) * (K + 1) + lane] : 0.f;
  const float uK = uniforms[static_cast<size_t>(b) * (K + 1) + K];
  // row statistics (nrows <= 2 SV_MAX_K + 1 = 65: rows lane, lane + 32, lane + 64)
  int err = 0;
#pragma unroll
  for (int t = 0; t < 3; ++t) {
    const int j = lane + 32 * t;
    if (j < nrows) {
      const float2 v = topk_mz[r0 + j];
      if (v.x != v.x) err |= 0x02;
      else if (v.x == kNegInf || !(v.y > 0.f)) err |= 0x04;
      wf.rm[j] = v.x;
      wf.rz[j] = v.y;
    }
  }
  // slot of x_i in p_i's list (ridx[2i]) and in q_i's (ridx[2i+1]), -1 if
  // absent: every (list, slot) pair is checked by some lane, eight loads in
  // flight at a time
  for (int i = lane; i < 2 * nd; i += 32) wf.ridx[i] = -1;
  __syncwarp();
  const int total = 2 * nd * k;
  for (int e0 = 0; e0 < total; e0 += 32 * 8) {
    int idv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u * 32 + lane;
      idv[u] = -1;
      if (e < total) {
        const int which = e / (nd * k), rem = e % (nd * k), i = rem / k, slot = rem % k;
        idv[u] = __float_as_int(list_of(which ? nd + 1 + i : i)[slot].y);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u * 32 + lane;
      if (e < total) {
        const int which = e / (nd * k), rem = e % (nd * k), i = rem / k, slot = rem % k;
        if (idv[u] >= 0 && idv[u] == tokens[static_cast<size_t>(b) * K + i])
          wf.ridx[2 * i + which] = slot;
      }
    }
  }
  __syncwarp();

  // accept tests (lane i = draft i), as in the unfiltered finalize
  bool acc = false;
  const double cd = static_cast<double>(c.hi) + static_cast<double>(c.lo);
  if (lane < nd) {
    if (x < 0 || x >= V) {
      err |= 0x01;
    } else {
      const int sp = wf.ridx[2 * lane], sq = wf.ridx[2 * lane + 1];
      const int jt = lane, jd = nd + 1 + lane;
      double np = 0.0, nq = 0.0;
      if (sp >= 0)
        np = exp2_nonpos((static_cast<double>(list_of(jt)[sp].x) -
                          static_cast<double>(wf.rm[jt])) * cd);
      if (sq >= 0)
        nq = exp2_nonpos((static_cast<double>(list_of(jd)[sq].x) -
                          static_cast<double>(wf.rm[jd])) * cd);
      const double zp = static_cast<double>(wf.rz[jt]), zq = static_cast<double>(wf.rz[jd]);
      acc = static_cast<double>(ui) * nq * zp < np * zq;
      if (!err) {
        if (p_at) p_at[static_cast<size_t>(b) * K + lane] = static_cast<float>(np) * rcp_fma(wf.rz[jt]);
        if (q_at) q_at[static_cast<size_t>(b) * K + lane] = static_cast<float>(nq) * rcp_fma(wf.rz[jd]);
      }
    }
  }
  err = __reduce_or_sync(0xffffffffu, err);
  for (int i = lane; i < K; i += 32) {
    if (err || i >= nd) {
      if (p_at) p_at[static_cast<size_t>(b) * K + i] = __int_as_float(0x7fc00000);
      if (q_at) q_at[static_cast<size_t>(b) * K + i] = __int_as_float(0x7fc00000);
    }
  }
  const unsigned mask = __ballot_sync(0xffffffffu, acc);
  int n = mask == 0xffffffffu ? 32 : __ffs(~mask) - 1;
  n = min(n, nd);

  // the draw over p_n's list: lane l holds slots 2l and 2l+1 (token order);
  // for the residual, q_n's logit of the same token if it is in q_n's list
  int token = -1;
  if (!err) {
    const int mode0 = n < nd ? 0 : 1;
    const int jp = n, jq = nd + 1 + n;
    float pv[2], xq[2];
    int pid[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int slot = 2 * lane + t;
      const float2 a = slot < k ? list_of(jp)[slot] : make_float2(kNegInf, __int_as_float(-1));
      pv[t] = a.x;
      pid[t] = __float_as_int(a.y);
      xq[t] = kNegInf;
    }
    if (mode0 == 0) {
      // q_n's list, slots lane and lane + 32, searched by every lane
      float qv[2];
      int qid[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int slot = lane + 32 * t;
        const float2 q = slot < k ? list_of(jq)[slot] : make_float2(kNegInf, __int_as_float(-1));
        qv[t] = q.x;
        qid[t] = __float_as_int(q.y);
      }
      for (int s2 = 0; s2 < 64; ++s2) {
        const int src = s2 & 31, tt = s2 >> 5;
        const int id2 = __shfl_sync(0xffffffffu, tt ? qid[1] : qid[0], src);
        const float v2 = __shfl_sync(0xffffffffu, tt ? qv[1] : qv[0], src);
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (id2 >= 0 && id2 == pid[t]) xq[t] = v2;
      }
    }
    const float mp = wf.rm[jp], izp = rcp_fma(wf.rz[jp]);
    const float mq = mode0 == 0 ? wf.rm[jq] : 0.f, izq = mode0 == 0 ? rcp_fma(wf.rz[jq]) : 0.f;
    for (int attempt = 0; attempt < 2 && token < 0; ++attempt) {
      // attempt 1: a residual of zero mass (rounding only) draws from p_n
      if (attempt == 1 && mode0 != 0) break;
      const int mode = attempt == 0 ? mode0 : 1;
      const ResidParams rp{mp, izp, mode == 0 ? mq : 0.f, mode == 0 ? izq : 0.f, c, mode};
      float w[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) w[t] = pid[t] >= 0 ? resid_weight(pv[t], xq[t], rp) : 0.f;
      // float-pair running sums in token order
      const DF incl = warp_incl_scan_df(df_add(df_add(DF{0.f, 0.f}, w[0]), w[1]), lane);
      const DF S = df_shfl(incl, 31);
      if (!(S.hi > 0.f)) continue;
      const DF target = df_mul(uK, S);
      DF excl = df_shfl(incl, lane > 0 ? lane - 1 : 0);
      if (lane == 0) excl = DF{0.f, 0.f};
      const DF e1 = df_add(excl, w[0]);
      // the first slot (token order) whose running sum exceeds target
      const bool h0 = w[0] > 0.f && df_lt(target, e1);
      const bool h1 = !h0 && w[1] > 0.f && df_lt(target, df_add(e1, w[1]));
      const unsigned hit = __ballot_sync(0xffffffffu, h0 || h1);
      if (hit) {
        const int src = __ffs(hit) - 1;
        token = __shfl_sync(0xffffffffu, h0 ? pid[0] : pid[1], src);
      } else {
        // rounding left target at the end: the last slot with weight
        const int lastp = w[1] > 0.f ? 1 : (w[0] > 0.f ? 0 : -1);
        const unsigned anyp = __ballot_sync(0xffffffffu, lastp >= 0);
        if (anyp) {
          const int src = 31 - __clz(anyp);
          token = __shfl_sync(0xffffffffu, lastp == 1 ? pid[1] : pid[0], src);
        }
      }
    }
    if (token < 0) err |= 0x04;
  }

  // outputs
  for (int i = lane; i <= K; i += 32) {
    int v = -1;
    if (!err) {
      if (i < n) v = tokens[static_cast<size_t>(b) * K + i];
      else if (i == n) v = token;
    }
    out_tokens[static_cast<size_t>(b) * (K + 1) + i] = v;
  }
  if (lane == 0) {
    out_len[b] = err ? 0 : n + 1;
    accept_len[b] = err ? 0 : n;
    if (err) record_error(&ws.hdr->error, err);
  }
  __syncwarp();
  // leave the lists and (m, Z) of the request's rows zero (see draw_finalize)
  for (int j = 0; j < nrows; ++j) {
    float2* l = const_cast<float2*>(list_of(j));
    for (int i = lane; i < max_topk; i += 32) l[i] = make_float2(0.f, 0.f);
  }
  for (int j = lane; j < nrows; j += 32) const_cast<float2*>(topk_mz)[r0 + j] = make_float2(0.f, 0.f);
  __syncwarp();
}

}  // namespace sv
