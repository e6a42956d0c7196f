// sv_tree.cuh -- token-tree verification.
//
// The tree of each request is depth-first linearised with parent indices
// (CMU 15-779 Lecture 17 notes, "Speculative Decoding", sec. 4.3).  The row
// pass reduces every node's target row and every draft row some node refers
// to; the finalize walks the tree from the root: VerifyGreedy for t == 0
// (sec. 4.4), multi-step speculative sampling for t > 0 (sec. 4.5):
// children are tried in ascending index order against the residual r
// (initially p_node), accept c iff u_c * q_c(x_c) < r(x_c), otherwise
// r <- norm(max(0, r - q_c)); all rejected -> draw from r; a leaf -> draw
// from p_node.  The residual lives in a per-request fp32 row of the
// workspace (unnormalised, with its fp64 total).
//
// Two more stochastic rules (greedy walks do not depend on them):
//   without replacement (children drawn without replacement; sec. 4.5 on
//     the proof's precondition, sec. 10 exercise 7): the j-th child tried
//     at a node is tested, and the residual formed, with q_j = q with the
//     tokens of the siblings tried before it removed and renormalised:
//     q_j(x) = q(x) / (1 - R) off the removed set (R = their q mass), 0 on
//     it.  The residual pass uses the scaled q everywhere and then puts
//     back r(y) at the removed tokens y.
//   naive sampling (sec. 4.5): draw x from p_node with u_accept[node]; move
//     to the first child whose token is x, else emit x.  No draft row is
//     read.
#pragma once

#include "sv_kernel.cuh"

namespace sv {

constexpr int kTreeMss = 0;
constexpr int kTreeNoReplace = 1;
constexpr int kTreeNaive = 2;

struct TreeProblem {
  static constexpr int kAuxBytes = 8;
  static constexpr bool kWarpFinalize = false;
  static constexpr bool kHasDraws = false;
  static constexpr bool kHasDirectFin = false;
  static constexpr bool kCtrl = false;
  int n_req, N, M, V, max_depth, es, ipr, chunk_el, max_topk;
  int mode;          // kTreeMss, kTreeNoReplace or kTreeNaive
  bool bulk;
  const char* target;
  int64_t t_stride;
  const char* draft;
  int64_t d_stride;
  const int* tokens;
  const int* parent;
  const int* q_row;
  const int* num_nodes;
  const float* temperature;
  const int* top_k;
  const float* u_accept;
  const float* u_sample;
  int* out_tokens;
  int* out_len;
  int* accept_len;
  int* accepted_nodes;
  Ws ws;

  __device__ int classify(int b, int& nn) const {
    nn = num_nodes ? num_nodes[b] : N;
    const float t = temperature[b];
    const int tk = top_k ? top_k[b] : 0;
    const bool filtered = tk > 0 && tk < V;
    if (nn < 1 || nn > N || !(t >= 0.f) || tk < 0) return -1;
    if (t == 0.f) return KIND_ARGMAX;
    if ((draft == nullptr && nn > 1 && mode != kTreeNaive) || filtered)
      return -1;  // top-k trees: not supported
    return KIND_SOFTMAX;
  }

  // draft rows referenced by nodes 1..nn-1 (bit m = draft row m)
  __device__ unsigned long long ref_mask(int b, int nn) const {
    unsigned long long m = 0ull;
    if (mode == kTreeNaive) return m;  // naive sampling reads no draft row
    for (int c = 1; c < nn; ++c) {
      const int r = q_row[static_cast<size_t>(b) * N + c];
      if (r >= 0 && r < M) m |= 1ull << r;
    }
    return m;
  }

  __device__ void write_failed(int b, int flag) const {
    for (int i = 0; i <= max_depth; ++i)
      out_tokens[static_cast<size_t>(b) * (max_depth + 1) + i] = -1;
    for (int i = 0; i < max_depth; ++i)
      accepted_nodes[static_cast<size_t>(b) * max_depth + i] = -1;
    out_len[b] = 0;
    accept_len[b] = 0;
    record_error(&ws.hdr->error, flag);
  }

  __device__ void prefetch_args(int) const {}

  __device__ void preamble(Shared& sh, PosTables& tab, int4* scan_tmp, unsigned char*) const {
    const int per = (n_req + kThreads - 1) / kThreads;
    const int lo = min(static_cast<int>(threadIdx.x) * per, n_req);
    const int hi = min(lo + per, n_req);
    int4 cnt = make_int4(0, 0, 0, 0);  // sampled n, sampled rows, other n, other rows
    for (int b = lo; b < hi; ++b) {
      int nn;
      const int kind = classify(b, nn);
      if (kind < 0) {
        cnt.z += 1;
      } else if (kind == KIND_ARGMAX) {
        cnt.z += 1;
        cnt.w += nn;
      } else {
        cnt.x += 1;
        cnt.y += nn + __popcll(ref_mask(b, nn));
      }
    }
    int4 tot;
    const int4 ex = block_excl_scan4(cnt, scan_tmp, tot);
    int hpos = ex.x, hrow = ex.y, lpos = tot.x + ex.z, lrow = tot.y + ex.w;
    for (int b = lo; b < hi; ++b) {
      int nn;
      const int kind = classify(b, nn);
      int pos;
      unsigned long long mask = 0ull;
      if (kind == KIND_SOFTMAX) {
        mask = ref_mask(b, nn);
        pos = hpos++;
        tab.rstart[pos] = hrow;
        hrow += nn + __popcll(mask);
      } else {
        pos = lpos++;
        tab.rstart[pos] = lrow;
        lrow += kind < 0 ? 0 : nn;
      }
      tab.info[pos] = make_info(b, kind < 0 ? 0 : kind, kind < 0 ? 0 : nn);
      reinterpret_cast<unsigned long long*>(tab.aux)[pos] = mask;
      const Scale2 c = scale_for(temperature[b]);
      tab.scale[pos] = make_float2(c.hi, c.lo);
      if (kind < 0 && blockIdx.x == 0) write_failed(b, 0x20);
    }
    if (threadIdx.x == 0) {
      tab.rstart[n_req] = tot.y + tot.w;
      sh.n_pos = n_req;
    }
  }

  __device__ void fill_stage(const PosTables& tab, int rl, StageMeta& mt, ResMeta& rm) const {
    const int info = tab.info[mt.pos];
    const int b = info_req(info), nn = info_extra(info);
    mt.kind = info_kind(info);
    const float2 s = tab.scale[mt.pos];
    mt.c_hi = s.x;
    mt.c_lo = s.y;
    const char* rp;
    if (rl < nn) {
      rp = target + (static_cast<int64_t>(b) * N + rl) * t_stride;
    } else {
      // the (rl - nn)-th referenced draft row
      unsigned long long m = ref_of(tab, mt.pos);
      for (int k = rl - nn; k > 0; --k) m &= m - 1;
      const int r = __ffsll(static_cast<long long>(m)) - 1;
      rp = draft + (static_cast<int64_t>(b) * M + r) * d_stride;
    }
    mt.src = rp + static_cast<size_t>(mt.el_base) * es;
    rm.tkt = b;
    rm.need = (tab.rstart[mt.pos + 1] - tab.rstart[mt.pos]) * ipr;
    rm.fin_code = mt.pos;
  }

  // trees draw inside their walk: no separate draw pass

  __device__ float4 consume(const StageMeta& mt, const unsigned char* sp, uint64_t* empty_bar,
                            int ctid, int lane) const {
    const float2 r = reduce_row_chunk(mt, sp, empty_bar, ctid, lane, bulk, es);
    return make_float4(r.x, r.y, 0.f, 0.f);
  }

  __device__ static unsigned long long ref_of(const PosTables& tab, int pos) {
    return reinterpret_cast<const unsigned long long*>(tab.aux)[pos];
  }

  __device__ void finalize(Shared& sh, const PosTables& tab, int pos, int ftid) const;
  __device__ void finalize_warp(Shared&, const PosTables&, int, int, WarpFin&) const {}
};

// Weights for the tree's inverse-CDF draw: either p_node (unnormalised
// 2^((l - m) c)) or the stored residual row.
struct TreeWeights {
  const char* prow;   // nullptr: read the stored residual
  const float* wrow;
  float mp;
  Scale2 c;
  int es, V;
  bool vec_ok;
  __device__ void operator()(int i0, float* w) const {
    if (prow != nullptr) {
      float x[32];
      load32(prow, es, vec_ok, i0, V, x);
#pragma unroll
      for (int j = 0; j < 32; ++j) w[j] = fast_exp2(scaled_arg(x[j], mp, c));
      return;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) w[j] = (i0 + j < V) ? wrow[i0 + j] : 0.f;
  }
};

__device__ void TreeProblem::finalize(Shared& sh, const PosTables& tab, int pos,
                                      int ftid) const {
  FinScratch& fs = sh.fin;
  const int warp = ftid >> 5, lane = ftid & 31;
  const int info = tab.info[pos];
  const int b = info_req(info), kind = info_kind(info), nn = info_extra(info);
  const unsigned long long mask = ref_of(tab, pos);
  const int r0 = tab.rstart[pos];
  const int nrows = tab.rstart[pos + 1] - r0;
  const Scale2 c{tab.scale[pos].x, tab.scale[pos].y};
  const bool greedy = kind == KIND_ARGMAX;
  const double cd = static_cast<double>(c.hi) + static_cast<double>(c.lo);
  const int* tok = tokens + static_cast<size_t>(b) * N;
  const int* par = parent + static_cast<size_t>(b) * N;
  const int* qr = q_row + static_cast<size_t>(b) * N;

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
  if (ftid == 0) fs.err = 0;
  named_sync(1, kFinThreads);

  // (2) validate the tree and the row statistics
  {
    int err = 0;
    for (int cc = ftid; cc < nn; cc += kFinThreads) {
      if (cc == 0) {
        if (par[0] != -1) err |= 0x08;
        continue;
      }
      const int p = par[cc];
      if (p < 0 || p >= cc) {
        err |= 0x08;
        continue;
      }
      if (tok[cc] < 0 || tok[cc] >= V) err |= 0x01;
      if (!greedy && mode != kTreeNaive && (qr[cc] < 0 || qr[cc] >= M)) err |= 0x08;
      int d = 0, x = cc;
      while (x > 0 && d <= max_depth) {
        const int px = par[x];
        if (px < 0 || px >= x) break;
        x = px;
        ++d;
      }
      if (d > max_depth) err |= 0x08;
    }
    for (int j = ftid; j < nrows; j += kFinThreads) {
      if (fs.rm[j] != fs.rm[j]) err |= 0x02;
      else if (fs.rm[j] == kNegInf || (!greedy && !(fs.rz[j] > 0.f))) err |= 0x04;
    }
    if (err) atomicOr(&fs.err, err);
  }
  named_sync(1, kFinThreads);
  int err = fs.err;

  int L = 0, node = 0, token = -1;
  __shared__ int children[SV_MAX_TREE_NODES];
  __shared__ int path[SV_MAX_TREE_NODES];
  __shared__ int n_children;
  __shared__ int decision;
  __shared__ double s_w;
  __shared__ int w_mode;  // 0: r = p_node, 1: r = stored residual row w_cur / s_w
  __shared__ int w_cur;   // which of the two residual rows holds r
  __shared__ double q_scale;  // 1 / (1 - removed q mass) (without replacement)
  while (!err) {
    // children of `node` in ascending index order
    if (warp == 0) {
      int cnt = 0;
      for (int base = node + 1; base < nn; base += 32) {
        const int cc = base + lane;
        const bool is_child = cc < nn && par[cc] == node;
        const unsigned bal = __ballot_sync(0xffffffffu, is_child);
        if (is_child) children[cnt + __popc(bal & ((1u << lane) - 1u))] = cc;
        cnt += __popc(bal);
      }
      if (lane == 0) {
        n_children = cnt;
        w_mode = 0;
        w_cur = 0;
        s_w = 0.0;
      }
    }
    named_sync(1, kFinThreads);
    const int nc = n_children;
    if (greedy) {
      const int a = fs.ridx[node];
      int next = -1;
      for (int k = 0; k < nc; ++k)
        if (tok[children[k]] == a) {
          next = children[k];
          break;
        }
      if (next < 0) {
        token = a;
        break;
      }
      if (ftid == 0) path[L] = next;
      ++L;
      node = next;
      named_sync(1, kFinThreads);
      continue;
    }
    const char* prow = target + (static_cast<int64_t>(b) * N + node) * t_stride;
    const float mp = fs.rm[node], zp = fs.rz[node];
    if (mode == kTreeNaive) {
      // naive sampling: a draw from p_node with the node's own uniform
      TreeWeights wp;
      wp.prow = prow;
      wp.wrow = nullptr;
      wp.mp = mp;
      wp.c = c;
      wp.es = es;
      wp.V = V;
      wp.vec_ok = bulk;
      const int x = icdf_draw(V, static_cast<double>(u_accept[static_cast<size_t>(b) * N + node]),
                              wp, fs, ftid);
      if (x < 0) {
        err |= 0x04;
        break;
      }
      int next = -1;
      for (int k = 0; k < nc; ++k)
        if (tok[children[k]] == x) {
          next = children[k];
          break;
        }
      if (next < 0) {
        token = x;
        break;
      }
      if (ftid == 0) path[L] = next;
      ++L;
      node = next;
      named_sync(1, kFinThreads);
      continue;
    }
    int next = -1;
    for (int k = 0; k < nc; ++k) {
      const int ch = children[k];
      const int qi = qr[ch];
      const int jq = nn + __popcll(mask & ((1ull << qi) - 1ull));
      const char* qrow = draft + (static_cast<int64_t>(b) * M + qi) * d_stride;
      const float mq = fs.rm[jq], zq = fs.rz[jq];
      const float* wsrc = ws.scratch + (static_cast<size_t>(b) * 2 + w_cur) * V;
      float* wdst = ws.scratch + (static_cast<size_t>(b) * 2 + (w_cur ^ 1)) * V;
      if (ftid == 0) {
        // without replacement: q_j = q off the earlier siblings' tokens,
        // scaled by 1 / (1 - R), R = their (distinct) q mass
        double qs = 1.0;
        bool removed = false;
        if (mode == kTreeNoReplace && k > 0) {
          double R = 0.0;
          for (int j = 0; j < k; ++j) {
            const int y = tok[children[j]];
            bool dup = false;
            for (int i = 0; i < j; ++i) dup |= tok[children[i]] == y;
            if (dup) continue;
            removed |= y == tok[ch];
            R += exp2(static_cast<double>(load_logit(qrow, es, y) - mq) * cd) /
                 static_cast<double>(zq);
          }
          qs = R < 1.0 ? 1.0 / (1.0 - R) : 0.0;
        }
        q_scale = qs;
        // accept test of child ch against the current residual r
        const int x = tok[ch];
        const double q = removed ? 0.0
                                 : exp2(static_cast<double>(load_logit(qrow, es, x) - mq) * cd) /
                                       static_cast<double>(zq) * qs;
        const double r =
            w_mode == 0
                ? exp2(static_cast<double>(load_logit(prow, es, x) - mp) * cd) /
                      static_cast<double>(zp)
                : static_cast<double>(__ldcg(wsrc + x)) / s_w;
        const double u = static_cast<double>(u_accept[static_cast<size_t>(b) * N + ch]);
        decision = u * q < r;
      }
      named_sync(1, kFinThreads);
      if (decision) {
        next = ch;
        break;
      }
      // rejected: r <- max(0, r - q_ch) into the other residual row
      const float izq = 1.f / zq, izp = 1.f / zp;
      const float inv_sw = w_mode == 0 ? 0.f : static_cast<float>(1.0 / s_w);
      const float qsf = static_cast<float>(q_scale);
      const int rmode = w_mode;
      auto r_at = [&](int t) {
        return rmode == 0 ? fast_exp2(scaled_arg(load_logit(prow, es, t), mp, c)) * izp
                          : __ldcg(wsrc + t) * inv_sw;
      };
      float part = 0.f;
      for (int t = ftid; t < V; t += kFinThreads) {
        const float rt = r_at(t);
        const float qt = fast_exp2(scaled_arg(load_logit(qrow, es, t), mq, c)) * izq * qsf;
        const float wt = fmaxf(rt - qt, 0.f);
        part += wt;
        __stcg(wdst + t, wt);
      }
      double dp = static_cast<double>(part);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dp += __shfl_xor_sync(0xffffffffu, dp, o);
      if (lane == 0) fs.dsum[warp] = dp;
      named_sync(1, kFinThreads);
      if (ftid == 0) {
        double S = 0.0;
        for (int w = 0; w < kFinWarps; ++w) S += fs.dsum[w];
        if (mode == kTreeNoReplace) {
          // q_j is 0 on the removed tokens: the residual there is r itself
          for (int j = 0; j < k; ++j) {
            const int y = tok[children[j]];
            bool dup = false;
            for (int i = 0; i < j; ++i) dup |= tok[children[i]] == y;
            if (dup) continue;
            const float ry = r_at(y);
            S += static_cast<double>(ry) - static_cast<double>(__ldcg(wdst + y));
            __stcg(wdst + y, ry);
          }
        }
        if (S > 0.0) {  // zero mass (rounding only) keeps r as it was
          s_w = S;
          w_mode = 1;
          w_cur ^= 1;
        }
      }
      named_sync(1, kFinThreads);
    }
    if (next >= 0) {
      if (ftid == 0) path[L] = next;
      ++L;
      node = next;
      named_sync(1, kFinThreads);
      continue;
    }
    // a leaf, or every child rejected: draw from r with u_sample
    TreeWeights wf;
    wf.prow = w_mode == 0 ? prow : nullptr;
    wf.wrow = ws.scratch + (static_cast<size_t>(b) * 2 + w_cur) * V;
    wf.mp = mp;
    wf.c = c;
    wf.es = es;
    wf.V = V;
    wf.vec_ok = bulk;
    token = icdf_draw(V, static_cast<double>(u_sample[b]), wf, fs, ftid);
    if (token < 0) err |= 0x04;
    break;
  }

  // outputs
  for (int i = ftid; i <= max_depth; i += kFinThreads) {
    int v = -1;
    if (!err) {
      if (i < L) v = tok[path[i]];
      else if (i == L) v = token;
    }
    out_tokens[static_cast<size_t>(b) * (max_depth + 1) + i] = v;
  }
  for (int i = ftid; i < max_depth; i += kFinThreads)
    accepted_nodes[static_cast<size_t>(b) * max_depth + i] = (!err && i < L) ? path[i] : -1;
  if (ftid == 0) {
    out_len[b] = err ? 0 : L + 1;
    accept_len[b] = err ? 0 : L;
    if (err) record_error(&ws.hdr->error, err);
    ws.tickets[b] = 0u;
  }
  // leave the request's chunk partials and residual rows zero: any part of
  // the workspace may serve a later chain call's partials, which must start
  // at zero
  for (int i = ftid; i < nrows * ipr; i += kFinThreads)
    ws.partials[static_cast<size_t>(r0) * ipr + i] = make_float2(0.f, 0.f);
  if (!greedy) {
    float* wrow = ws.scratch + static_cast<size_t>(b) * 2 * V;
    for (int i = ftid; i < 2 * V; i += kFinThreads) wrow[i] = 0.f;
  }
  named_sync(1, kFinThreads);
}

}  // namespace sv
