// sv_resid.cuh -- the residual / bonus draw of sampled chain requests,
// spread over the whole GPU.
//
// After the accept scan of a sampled request stops at position n, one token
// is drawn by inverse CDF from w = max(0, p_n - q_n) (rejection) or from
// w = p_n (every draft accepted) -- CMU 15-779 Lecture 17 notes,
// "Speculative Decoding", sec. 2.3-2.4; study notes "LLM speculative
// decoding 02", sec. 4.  The chain finalize leaves one job per such request;
// this pass splits each job's row pair into chunks of 8192 (bf16) or 4096
// (fp32) tokens, staged as p-chunk | q-chunk in one 32 KB stage.  Each
// consumer warp turns its 1/16 of a chunk (one "segment") into residual
// weights and their sum; the request's last arriving chunk hands the job to
// a finalize that takes the fp64 prefix over the segment sums, finds the
// segment holding u * S and rescans just that segment with bit-identical
// arithmetic to pick the token.
#pragma once

#include "sv_kernel.cuh"

namespace sv {


struct ResidJob {
  int b, n, mode;  // mode 0: residual max(0, p_n - q_n); 1: bonus p_n
  float mp, izp, mq, izq;
  float c_hi, c_lo;
  int pad[3];
};

struct ResidParams {
  float mp, izp, mq, izq;
  Scale2 c;
  int mode;
};

// Residual weight of one token from its two logits.  Every operation is an
// explicitly rounded intrinsic, so the chunk pass and the final rescan
// produce the same bits.
__device__ __forceinline__ float resid_weight(float xp, float xq, const ResidParams& r) {
  const float dp = fmaxf(__fsub_rn(xp, r.mp), -1.0e30f);
  const float ep = fast_exp2(__fmaf_rn(dp, r.c.hi, __fmul_rn(dp, r.c.lo)));
  if (r.mode != 0) return ep;  // bonus: unnormalised p
  const float dq = fmaxf(__fsub_rn(xq, r.mq), -1.0e30f);
  const float eq = fast_exp2(__fmaf_rn(dq, r.c.hi, __fmul_rn(dq, r.c.lo)));
  return fmaxf(__fsub_rn(__fmul_rn(ep, r.izp), __fmul_rn(eq, r.izq)), 0.f);
}

__device__ __forceinline__ float warp_incl_scan_rn(float x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = __fadd_rn(x, y);
  }
  return x;
}

struct ResidProblem {
  static constexpr int kAuxBytes = 16;
  int n_req, K, V, es, ipr, chunk_el;
  bool bulk;
  const char* target;
  int64_t t_stride;
  const char* draft;
  int64_t d_stride;
  const float* uniforms;
  int* out_tokens;
  int* out_len;
  int* accept_len;
  const ResidJob* jobs;
  Ws ws;

  __device__ int seg_el() const { return chunk_el / kConsumerWarps; }

  // one position per job, one "row" (the row pair) per position
  __device__ void preamble(Shared& sh, PosTables& tab, int4*) const {
    const int n_jobs = min(static_cast<int>(*reinterpret_cast<volatile int*>(&ws.hdr->n_jobs)), n_req);
    for (int j = threadIdx.x; j < n_jobs; j += kThreads) {
      const ResidJob jb = jobs[j];
      tab.info[j] = make_info(jb.b, jb.mode, jb.n);
      tab.rstart[j] = j;
      tab.scale[j] = make_float2(jb.c_hi, jb.c_lo);
      tab.aux[j] = make_float4(jb.mp, jb.izp, jb.mq, jb.izq);
    }
    if (threadIdx.x == 0) {
      tab.rstart[n_jobs] = n_jobs;
      sh.n_pos = n_jobs;
    }
  }

  __device__ const char* prow(int b, int n) const {
    return target + (static_cast<int64_t>(b) * (K + 1) + n) * t_stride;
  }
  __device__ const char* qrow(int b, int n) const {
    return draft + (static_cast<int64_t>(b) * K + n) * d_stride;
  }

  __device__ void fill_stage(const PosTables& tab, int, StageMeta& mt) const {
    const int info = tab.info[mt.pos];
    const int b = info_req(info), mode = info_kind(info), n = info_extra(info);
    mt.kind = KIND_RESID_PASS;
    const float2 s = tab.scale[mt.pos];
    mt.c_hi = s.x;
    mt.c_lo = s.y;
    mt.aux = tab.aux[mt.pos];
    mt.src = prow(b, n) + static_cast<size_t>(mt.el_base) * es;
    mt.src2 = mode == 0 ? qrow(b, n) + static_cast<size_t>(mt.el_base) * es : nullptr;
    mt.sub = mode;
  }

  // The warp's segment: elements [warp*seg, (warp+1)*seg) of the chunk, lane
  // l takes `per` consecutive ones; returns (segment sum, 0).
  __device__ float2 consume(const StageMeta& mt, const unsigned char* sp, uint64_t* empty_bar,
                            int ctid, int lane) const {
    const int warp = ctid >> 5;
    const int seg = seg_el(), per = seg / 32;
    const int e0 = warp * seg + lane * per;
    const int mode = mt.sub;
    float xp[16], xq[16];
    const char* pb = bulk ? reinterpret_cast<const char*>(sp) : mt.src;
    const char* qb = bulk ? reinterpret_cast<const char*>(sp) + kChunkBytes / 2 : mt.src2;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j < per) {
        const int e = e0 + j;
        const bool in = e < mt.n_el;
        xp[j] = in ? load_logit(pb, es, e) : kNegInf;
        xq[j] = (in && mode == 0) ? load_logit(qb, es, e) : kNegInf;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar);
    const ResidParams r{mt.aux.x, mt.aux.y, mt.aux.z, mt.aux.w, Scale2{mt.c_hi, mt.c_lo}, mode};
    float ls = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < per && e0 + j < mt.n_el) ls = __fadd_rn(ls, resid_weight(xp[j], xq[j], r));
    const float inc = warp_incl_scan_rn(ls, lane);
    return make_float2(__shfl_sync(0xffffffffu, inc, 31), 0.f);
  }

  __device__ void finalize(Shared& sh, const PosTables& tab, int pos, int ftid) const;

  // the last CTA of the pass clears the job count for the next call
  __device__ void last_cta_reset() const { ws.hdr->n_jobs = 0; }
};

__device__ void ResidProblem::finalize(Shared& sh, const PosTables& tab, int pos,
                                       int ftid) const {
  FinScratch& fs = sh.fin;
  const int warp = ftid >> 5, lane = ftid & 31;
  const int info = tab.info[pos];
  const int b = info_req(info), mode = info_kind(info), n = info_extra(info);
  const int seg = seg_el(), per = seg / 32;
  const int nseg = ipr * kConsumerWarps;
  const float2* segsum = ws.partials + static_cast<size_t>(pos) * ipr * kConsumerWarps;
  const double u = static_cast<double>(uniforms[static_cast<size_t>(b) * (K + 1) + K]);
  const float4 a = tab.aux[pos];
  const ResidParams rp{a.x, a.y, a.z, a.w, Scale2{tab.scale[pos].x, tab.scale[pos].y}, mode};
  const char* pr = prow(b, n);
  const char* qr = qrow(b, n);

  // fp64 prefix over the segment sums: thread t takes a contiguous block
  const int blk = (nseg + kFinThreads - 1) / kFinThreads;
  const int lo = min(ftid * blk, nseg), hi = min(lo + blk, nseg);
  double tsum = 0.0;
  for (int s = lo; s < hi; ++s) tsum += static_cast<double>(__ldcg(&segsum[s].x));
  double incl = warp_incl_scan_d(tsum, lane);
  if (lane == 31) fs.dsum[warp] = incl;
  named_sync(1, kFinThreads);
  double before = 0.0, S = 0.0;
  for (int w = 0; w < kFinWarps; ++w) {
    if (w < warp) before += fs.dsum[w];
    S += fs.dsum[w];
  }
  const double excl = before + incl - tsum;
  const double target = u * S;
  int found = -1, last_pos = -1;
  double base = 0.0, run = excl;
  for (int s = lo; s < hi; ++s) {
    const float v = __ldcg(&segsum[s].x);
    const double nxt = run + static_cast<double>(v);
    if (found < 0 && target < nxt) {
      found = s;
      base = run;
    }
    if (v > 0.f) last_pos = s;
    run = nxt;
  }
  if (ftid == 0) {
    fs.seg_k = 0x7fffffff;
    fs.seg_mode = -1;
  }
  named_sync(1, kFinThreads);
  if (S > 0.0) {
    if (found >= 0) atomicMin(&fs.seg_k, found);
    else if (last_pos >= 0) atomicMax(&fs.seg_mode, last_pos);
  }
  named_sync(1, kFinThreads);
  if (found >= 0 && found == fs.seg_k) fs.base = base;  // the thread that owns segment k
  named_sync(1, kFinThreads);

  int token = -1;
  const bool have_mass = S > 0.0 && (fs.seg_k != 0x7fffffff || fs.seg_mode >= 0);
  if (have_mass && warp == 0) {
    const bool exact = fs.seg_k != 0x7fffffff;  // else: take the last positive weight
    const int k = exact ? fs.seg_k : fs.seg_mode;
    // rescan segment k exactly as the chunk pass computed it
    const int e0 = (k / kConsumerWarps) * chunk_el + (k % kConsumerWarps) * seg + lane * per;
    float w[16];
    float ls = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      w[j] = 0.f;
      if (j < per && e0 + j < V) {
        const float xp = load_logit(pr, es, e0 + j);
        const float xq = mode == 0 ? load_logit(qr, es, e0 + j) : kNegInf;
        w[j] = resid_weight(xp, xq, rp);
        ls = __fadd_rn(ls, w[j]);
      }
    }
    const float inc = warp_incl_scan_rn(ls, lane);
    float exl = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) exl = 0.f;
    int tok = -1, src;
    if (exact) {
      const bool lane_hit = target < fs.base + static_cast<double>(inc);
      const unsigned lh = __ballot_sync(0xffffffffu, lane_hit);
      src = lh ? __ffs(lh) - 1 : 31;
      if (lane == src) {
        double c = fs.base + static_cast<double>(exl);
        int lastp = -1;
        for (int j = 0; j < per; ++j) {
          c += static_cast<double>(w[j]);
          if (w[j] > 0.f) lastp = j;
          if (tok < 0 && target < c) tok = j;
        }
        if (tok < 0) tok = lastp;
      }
    } else {
      int lastp = -1;
      for (int j = 0; j < per; ++j)
        if (w[j] > 0.f) lastp = j;
      const unsigned lp = __ballot_sync(0xffffffffu, lastp >= 0);
      src = lp ? 31 - __clz(lp) : 0;
      tok = lastp;
    }
    tok = __shfl_sync(0xffffffffu, tok, src);
    const int src_e0 = __shfl_sync(0xffffffffu, e0, src);
    if (lane == 0) fs.token = tok < 0 ? -1 : src_e0 + tok;
  }
  named_sync(1, kFinThreads);
  token = have_mass ? fs.token : -1;
  named_sync(1, kFinThreads);
  if (token < 0 && mode == 0) {
    // a residual of zero mass (rounding only): draw from p_n instead
    struct PWeights {
      const char* pr;
      ResidParams r;
      int es, V;
      __device__ void operator()(int i0, float* w) const {
        for (int j = 0; j < 32; ++j)
          w[j] = (i0 + j < V) ? resid_weight(load_logit(pr, es, i0 + j), kNegInf, r) : 0.f;
      }
    };
    ResidParams rb = rp;
    rb.mode = 1;
    token = icdf_draw(V, u, PWeights{pr, rb, es, V}, fs, ftid);
  }
  if (ftid == 0) {
    if (token >= 0) {
      out_tokens[static_cast<size_t>(b) * (K + 1) + n] = token;
    } else {
      for (int i = 0; i <= K; ++i) out_tokens[static_cast<size_t>(b) * (K + 1) + i] = -1;
      out_len[b] = 0;
      accept_len[b] = 0;
      record_error(&ws.hdr->error, 0x04);
    }
    ws.tickets[b] = 0u;
  }
  named_sync(1, kFinThreads);
}

}  // namespace sv
