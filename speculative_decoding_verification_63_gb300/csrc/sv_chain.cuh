// sv_chain.cuh -- chain verification (one chain of K drafts per request).
//
// The step follows Algorithm 1 as restated in the CMU 15-779 Lecture 17
// notes ("Speculative Decoding", sec. 2.4) and the study notes "LLM
// speculative decoding 02" (sec. 4): accept draft x_i iff
// u_i * q_i(x_i) < p_i(x_i), stop at the first rejection n, emit a draw
// from norm(max(0, p_n - q_n)) -- or, if all drafts pass, from p_{nd} --
// by inverse CDF with u_K.  Greedy requests (t == 0) accept iff x_i is the
// argmax of target row i (lecture notes sec. 2.2; study notes sec. 10).
#pragma once

#include "sv_resid.cuh"

namespace sv {

struct ChainProblem {
  static constexpr int kAuxBytes = 0;
  int n_req, K, V, es, ipr, chunk_el, max_topk;
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
  ResidJob* jobs;  // sampled requests leave their residual / bonus draw here
  Ws ws;

  // kind of request b, or -1 if its scalar arguments are invalid
  __device__ int classify(int b, int& nd) const {
    nd = num_drafts ? num_drafts[b] : K;
    const float t = temperature[b];
    const int tk = top_k ? top_k[b] : 0;
    const bool filtered = tk > 0 && tk < V;
    if (nd < 0 || nd > K || !(t >= 0.f) || tk < 0) return -1;
    if (t == 0.f) return KIND_ARGMAX;
    if ((draft == nullptr && nd > 0) || filtered) return -1;  // top-k: not yet supported
    return KIND_SOFTMAX;
  }

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

  // Processing order: sampled unfiltered requests first (their finalize
  // streams a row pair and should overlap the rest of the pass), then
  // filtered and greedy ones.  rows: greedy nd+1, sampled 2nd+1.
  __device__ void preamble(Shared& sh, PosTables& tab, int4* scan_tmp) const {
    const int per = (n_req + kThreads - 1) / kThreads;
    const int lo = min(static_cast<int>(threadIdx.x) * per, n_req);
    const int hi = min(lo + per, n_req);
    int4 cnt = make_int4(0, 0, 0, 0);  // heavy n, heavy rows, light n, light rows
    for (int b = lo; b < hi; ++b) {
      int nd;
      const int kind = classify(b, nd);
      if (kind < 0) {
        cnt.z += 1;
        continue;
      }
      const int rows = kind == KIND_ARGMAX ? nd + 1 : 2 * nd + 1;
      if (kind == KIND_SOFTMAX) {
        cnt.x += 1;
        cnt.y += rows;
      } else {
        cnt.z += 1;
        cnt.w += rows;
      }
    }
    int4 tot;
    const int4 ex = block_excl_scan4(cnt, scan_tmp, tot);
    int hpos = ex.x, hrow = ex.y, lpos = tot.x + ex.z, lrow = tot.y + ex.w;
    for (int b = lo; b < hi; ++b) {
      int nd;
      const int kind = classify(b, nd);
      int pos, rows = 0;
      if (kind == KIND_SOFTMAX) {
        rows = 2 * nd + 1;
        pos = hpos++;
        tab.rstart[pos] = hrow;
        hrow += rows;
      } else {
        rows = kind < 0 ? 0 : (kind == KIND_ARGMAX ? nd + 1 : 2 * nd + 1);
        pos = lpos++;
        tab.rstart[pos] = lrow;
        lrow += rows;
      }
      tab.info[pos] = make_info(b, kind < 0 ? 0 : kind, nd < 0 ? 0 : min(nd, 0x7ff));
      const Scale2 c = scale_for(temperature[b]);
      tab.scale[pos] = make_float2(c.hi, c.lo);
      if (kind < 0 && blockIdx.x == 0) write_failed(b, 0x20);
    }
    if (threadIdx.x == 0) {
      tab.rstart[n_req] = tot.y + tot.w;
      sh.n_pos = n_req;
    }
  }

  __device__ void fill_stage(const PosTables& tab, int rl, StageMeta& mt) const {
    const int info = tab.info[mt.pos];
    const int b = info_req(info), nd = info_extra(info);
    mt.kind = info_kind(info);
    const float2 s = tab.scale[mt.pos];
    mt.c_hi = s.x;
    mt.c_lo = s.y;
    const char* rp = rl <= nd ? target + (static_cast<int64_t>(b) * (K + 1) + rl) * t_stride
                              : draft + (static_cast<int64_t>(b) * K + (rl - nd - 1)) * d_stride;
    mt.src = rp + static_cast<size_t>(mt.el_base) * es;
  }

  __device__ float2 consume(const StageMeta& mt, const unsigned char* sp, uint64_t* empty_bar,
                            int ctid, int lane) const {
    return reduce_row_chunk(mt, sp, empty_bar, ctid, lane, bulk, es);
  }

  __device__ void finalize(Shared& sh, const PosTables& tab, int pos, int ftid) const;
  __device__ void last_cta_reset() const {}
};

// Residual / bonus weights of 32 consecutive tokens (tree walk helper).
struct ChainWeights {
  const char* prow;
  const char* qrow;  // nullptr: bonus mode, w = 2^((l - m_p) c)
  float mp, mq, izp, izq;
  Scale2 c;
  int es, V;
  bool vec_ok;
  __device__ void operator()(int i0, float* w) const {
    float x[32];
    load32(prow, es, vec_ok, i0, V, x);
    if (qrow == nullptr) {
#pragma unroll
      for (int j = 0; j < 32; ++j) w[j] = fast_exp2(scaled_arg(x[j], mp, c));
      return;
    }
    float y[32];
    load32(qrow, es, vec_ok, i0, V, y);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float pv = fast_exp2(scaled_arg(x[j], mp, c)) * izp;
      const float qv = fast_exp2(scaled_arg(y[j], mq, c)) * izq;
      w[j] = fmaxf(pv - qv, 0.f);
    }
  }
};

__device__ void ChainProblem::finalize(Shared& sh, const PosTables& tab, int pos,
                                       int ftid) const {
  FinScratch& fs = sh.fin;
  const int warp = ftid >> 5, lane = ftid & 31;
  const int info = tab.info[pos];
  const int b = info_req(info), kind = info_kind(info), nd = info_extra(info);
  const int r0 = tab.rstart[pos];
  const int nrows = tab.rstart[pos + 1] - r0;
  const Scale2 c{tab.scale[pos].x, tab.scale[pos].y};
  const bool greedy = kind == KIND_ARGMAX;

  // (1) merge the chunk partials of every row: a warp takes 32 / ipr rows
  // per pass, one group of ipr lanes per row (all loads issued first), then
  // a guarded shfl_down tree within each group
  {
    const int width = ipr <= 32 ? ipr : 32;
    const int rpw = 32 / width;
    const int g = lane / width, r = lane % width;
    for (int j0 = warp * rpw; j0 < nrows; j0 += kFinWarps * rpw) {
      const int j = j0 + g;
      const bool own = g < rpw && j < nrows;
      const float2* pp = ws.partials + static_cast<size_t>(r0 + (own ? j : 0)) * ipr;
      if (greedy) {
        VI v{kNegInf, 0x7fffffff};
        if (own)
          for (int ch = r; ch < ipr; ch += width) {
            const float2 u = __ldcg(pp + ch);
            v = vi_better(v, VI{u.x, __float_as_int(u.y)});
          }
        for (int o = 1; o < width; o <<= 1) {
          const VI w{__shfl_down_sync(0xffffffffu, v.v, o), __shfl_down_sync(0xffffffffu, v.i, o)};
          if (r + o < width) v = vi_better(v, w);
        }
        if (own && r == 0) {
          fs.rm[j] = v.v;
          fs.ridx[j] = v.i;
        }
      } else {
        MS v{kNegInf, 0.f};
        if (own)
          for (int ch = r; ch < ipr; ch += width) {
            const float2 u = __ldcg(pp + ch);
            v = ms_combine(v, MS{u.x, u.y}, c);
          }
        for (int o = 1; o < width; o <<= 1) {
          const MS w{__shfl_down_sync(0xffffffffu, v.m, o), __shfl_down_sync(0xffffffffu, v.s, o)};
          if (r + o < width) v = ms_combine(v, w, c);
        }
        if (own && r == 0) {
          fs.rm[j] = v.m;
          fs.rz[j] = v.s;
        }
      }
    }
  }
  named_sync(1, kFinThreads);

  // (2) accept tests and the prefix-terminating scan (warp 0, lane i = draft i)
  if (warp == 0) {
    int err = 0;
    bool acc = false;
    // every row must be finite and carry mass
    for (int j = lane; j < nrows; j += 32) {
      if (fs.rm[j] != fs.rm[j]) err |= 0x02;
      else if (fs.rm[j] == kNegInf || (!greedy && !(fs.rz[j] > 0.f))) err |= 0x04;
    }
    const double cd = static_cast<double>(c.hi) + static_cast<double>(c.lo);
    if (lane < nd) {
      const int x = tokens[static_cast<size_t>(b) * K + lane];
      if (x < 0 || x >= V) {
        err |= 0x01;
      } else if (greedy) {
        acc = x == fs.ridx[lane];
        if (p_at) p_at[static_cast<size_t>(b) * K + lane] = acc ? 1.f : 0.f;
        if (q_at) q_at[static_cast<size_t>(b) * K + lane] = __int_as_float(0x7fc00000);
      } else {
        const char* trow = target + (static_cast<int64_t>(b) * (K + 1) + lane) * t_stride;
        const char* drow = draft + (static_cast<int64_t>(b) * K + lane) * d_stride;
        const float lx = load_logit(trow, es, x), dx = load_logit(drow, es, x);
        const int jt = lane, jd = nd + 1 + lane;
        const double p = exp2(static_cast<double>(lx - fs.rm[jt]) * cd) /
                         static_cast<double>(fs.rz[jt]);
        const double q = exp2(static_cast<double>(dx - fs.rm[jd]) * cd) /
                         static_cast<double>(fs.rz[jd]);
        const double u = static_cast<double>(uniforms[static_cast<size_t>(b) * (K + 1) + lane]);
        acc = u * q < p;
        if (p_at) p_at[static_cast<size_t>(b) * K + lane] = static_cast<float>(p);
        if (q_at) q_at[static_cast<size_t>(b) * K + lane] = static_cast<float>(q);
      }
    } else if (lane < K) {
      if (p_at) p_at[static_cast<size_t>(b) * K + lane] = __int_as_float(0x7fc00000);
      if (q_at) q_at[static_cast<size_t>(b) * K + lane] = __int_as_float(0x7fc00000);
    }
    for (int i = 32 + lane; i < K; i += 32) {  // K <= 32 keeps this empty
      if (p_at) p_at[static_cast<size_t>(b) * K + i] = __int_as_float(0x7fc00000);
      if (q_at) q_at[static_cast<size_t>(b) * K + i] = __int_as_float(0x7fc00000);
    }
    err = __reduce_or_sync(0xffffffffu, err);
    const unsigned mask = __ballot_sync(0xffffffffu, acc);
    int n = mask == 0xffffffffu ? 32 : __ffs(~mask) - 1;
    n = min(n, nd);
    if (lane == 0) {
      fs.n_acc = n;
      fs.err = err;
    }
  }
  named_sync(1, kFinThreads);
  const int n = fs.n_acc;
  const int err = fs.err;

  // (3) the emitted token: greedy here; sampled requests hand the draw to
  // the residual pass (one job: row pair n, residual or bonus)
  int token = -1;
  const int err2 = err;
  if (!err && greedy) token = fs.ridx[n];
  if (!err && !greedy && ftid == 0) {
    const int jid = atomicAdd(&ws.hdr->n_jobs, 1);
    ResidJob jb;
    jb.b = b;
    jb.n = n;
    jb.mode = n < nd ? 0 : 1;
    jb.mp = fs.rm[n];
    jb.izp = 1.f / fs.rz[n];
    jb.mq = n < nd ? fs.rm[nd + 1 + n] : 0.f;
    jb.izq = n < nd ? 1.f / fs.rz[nd + 1 + n] : 0.f;
    jb.c_hi = c.hi;
    jb.c_lo = c.lo;
    jobs[jid] = jb;
  }

  // (4) outputs; reset this request's ticket for the next call
  if (ftid <= K) {
    int v = -1;
    if (!err2) {
      if (ftid < n) v = tokens[static_cast<size_t>(b) * K + ftid];
      else if (ftid == n) v = token;  // sampled: written by the residual pass
    }
    out_tokens[static_cast<size_t>(b) * (K + 1) + ftid] = v;
  }
  if (ftid == 0) {
    out_len[b] = err2 ? 0 : n + 1;
    accept_len[b] = err2 ? 0 : n;
    if (err2) record_error(&ws.hdr->error, err2);
    ws.tickets[b] = 0u;
  }
  named_sync(1, kFinThreads);
}

}  // namespace sv
