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

#include "sv_kernel.cuh"

namespace sv {

struct ChainProblem {
  static constexpr bool kAux = false;
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

  __device__ const char* row_ptr(const PosTables& tab, int pos, int rl, int& kind,
                                 Scale2& c) const {
    const int info = tab.info[pos];
    const int b = info_req(info), nd = info_extra(info);
    kind = info_kind(info);
    const float2 s = tab.scale[pos];
    c.hi = s.x;
    c.lo = s.y;
    if (rl <= nd) return target + (static_cast<int64_t>(b) * (K + 1) + rl) * t_stride;
    return draft + (static_cast<int64_t>(b) * K + (rl - nd - 1)) * d_stride;
  }

  __device__ void finalize(Shared& sh, const PosTables& tab, int pos, int ctid) const;
};

// Residual / bonus weights of 32 consecutive tokens.
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
                                       int ctid) const {
  FinScratch& fs = sh.fin;
  const int warp = ctid >> 5, lane = ctid & 31;
  const int info = tab.info[pos];
  const int b = info_req(info), kind = info_kind(info), nd = info_extra(info);
  const int r0 = tab.rstart[pos];
  const int nrows = tab.rstart[pos + 1] - r0;
  const Scale2 c{tab.scale[pos].x, tab.scale[pos].y};
  const bool greedy = kind == KIND_ARGMAX;

  // (1) merge the chunk partials of every row of this request
  for (int j = warp; j < nrows; j += kConsumerWarps) {
    const float2* pp = ws.partials + static_cast<size_t>(r0 + j) * ipr;
    if (greedy) {
      VI v{kNegInf, 0x7fffffff};
      for (int ch = lane; ch < ipr; ch += 32) {
        const float2 t = __ldcg(pp + ch);
        v = vi_better(v, VI{t.x, __float_as_int(t.y)});
      }
      v = warp_reduce_vi(v);
      if (lane == 0) {
        fs.rm[j] = v.v;
        fs.ridx[j] = v.i;
      }
    } else {
      MS v{kNegInf, 0.f};
      for (int ch = lane; ch < ipr; ch += 32) {
        const float2 t = __ldcg(pp + ch);
        v = ms_combine(v, MS{t.x, t.y}, c);
      }
      v = warp_reduce_ms(v, c);
      if (lane == 0) {
        fs.rm[j] = v.m;
        fs.rz[j] = v.s;
      }
    }
  }
  named_sync(1, kConsumers);

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
  named_sync(1, kConsumers);
  const int n = fs.n_acc;
  const int err = fs.err;

  // (3) the emitted token
  int token = -1;
  int err2 = err;
  if (!err) {
    if (greedy) {
      token = fs.ridx[n];
    } else {
      const double u = static_cast<double>(uniforms[static_cast<size_t>(b) * (K + 1) + K]);
      ChainWeights wf;
      wf.prow = target + (static_cast<int64_t>(b) * (K + 1) + n) * t_stride;
      wf.mp = fs.rm[n];
      wf.izp = 1.f / fs.rz[n];
      wf.c = c;
      wf.es = es;
      wf.V = V;
      wf.vec_ok = bulk;
      if (n < nd) {
        wf.qrow = draft + (static_cast<int64_t>(b) * K + n) * d_stride;
        wf.mq = fs.rm[nd + 1 + n];
        wf.izq = 1.f / fs.rz[nd + 1 + n];
      } else {
        wf.qrow = nullptr;
        wf.mq = 0.f;
        wf.izq = 0.f;
      }
      token = icdf_draw(V, u, wf, fs, ctid);
      if (token < 0 && wf.qrow != nullptr) {
        // residual of zero mass (rounding only): draw from p_n instead
        wf.qrow = nullptr;
        token = icdf_draw(V, u, wf, fs, ctid);
      }
      if (token < 0) err2 |= 0x04;
    }
  }

  // (4) outputs; reset this request's ticket for the next call
  if (ctid <= K) {
    int v = -1;
    if (!err2) {
      if (ctid < n) v = tokens[static_cast<size_t>(b) * K + ctid];
      else if (ctid == n) v = token;
    }
    out_tokens[static_cast<size_t>(b) * (K + 1) + ctid] = v;
  }
  if (ctid == 0) {
    out_len[b] = err2 ? 0 : n + 1;
    accept_len[b] = err2 ? 0 : n;
    if (err2) record_error(&ws.hdr->error, err2);
    ws.tickets[b] = 0u;
  }
  named_sync(1, kConsumers);
}

}  // namespace sv
