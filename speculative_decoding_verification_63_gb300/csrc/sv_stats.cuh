// sv_stats.cuh -- per-position acceptance statistics of a chain round.
//
// For position i of request b the acceptance probability of the draft is
// alpha_i = sum_x min(p_i(x), q_i(x)) = 1 - TV(p_i, q_i) (CMU 15-779
// Lecture 17 notes, "Speculative Decoding", sec. 2.3, Thm 3.5); with one
// rate per position the round emits sum_{j=0..nd} prod_{i<j} alpha_i tokens
// on average ("LLM speculative decoding study notes 02", sec. 7, where all
// rates are equal).  Greedy requests have one-hot p and q: alpha_i is 1 iff
// the two argmaxes (lowest id on ties) agree.
//
// alpha needs both rows normalised before the sum of minima, so every row
// pair is visited twice.  One cluster of kStCluster CTAs takes one pair:
// each CTA loads its 1/kStCluster of both rows into registers (16-byte
// streaming loads, all in flight together), reduces (max, sum) -- or the
// argmax -- over them, and the CTAs exchange their partials through
// distributed shared memory.  Every CTA merges the partials in rank order
// (so all agree bit for bit), and the second pass runs over the registers:
// min(p, q) = 2^min(a, b) with a = (l - M_p) c - log2 Z_p and likewise b,
// one exp2 per token instead of two.  Rank 0 adds the CTAs' sums in rank
// order.  HBM sees each row once; rows longer than the register tile
// (bf16 V > 131072, fp32 V > 65536) read their tail twice, the second time
// mostly from L2.
//
// The rank-0 CTA of the last pair of a request to finish (a counter per
// request in the workspace, reset afterwards) adds up the expected tokens.
//
// Sampled requests with a top-k filter ("LLM speculative decoding study
// notes 02", sec. 5.4: p and q each keep their own k most likely tokens)
// take another route: the chain's top-k pass (sv_topk.cuh) reduces their
// rows to (logit, id) lists and (m, Z), and row_stats_topk_kernel, one warp
// per request, sums min(p, q) over the tokens both lists hold -- elsewhere
// one of the two is zero.
#pragma once

#include <cooperative_groups.h>

#include "sv_rowpass.cuh"

namespace sv {

constexpr int kStCluster = 8;  // CTAs per row pair (portable cluster size)
constexpr int kStThreads = 256;
constexpr int kStWarps = kStThreads / 32;
constexpr int kStSlots = 8;    // 16-byte vectors per row a thread keeps in registers

struct StatsProblem {
  int B, K, V;
  int max_topk;      // bound on top_k with top-k lists in the workspace (0: none)
  bool vec;          // 16-byte aligned rows, strides and row lengths
  const char* target;
  int64_t t_stride;  // bytes
  const char* draft;
  int64_t d_stride;
  const int* num_drafts;
  const float* temperature;
  const int* top_k;
  float* alpha;
  float* expected;
  WsHeader* hdr;
  unsigned* tickets;
};

// What one CTA hands to the rest of its cluster.
struct StatsPart {
  float a0, a1, a2, a3;  // (m_p, s_p, m_q, s_q), or argmax (v_p, i_p, v_q, i_q)
  int flags;             // SV_DERR_NONFINITE when a NaN / +inf was seen
  double sum;            // the CTA's sum of min(p, q)
};

template <int ES>
__device__ __forceinline__ float vec_elem(const uint4& v, int j) {
  if constexpr (ES == 2) {
    const unsigned x = (j >> 1) == 0 ? v.x : (j >> 1) == 1 ? v.y : (j >> 1) == 2 ? v.z : v.w;
    return (j & 1) ? bf16hi(x) : bf16lo(x);
  } else {
    const unsigned x = j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
    return __uint_as_float(x);
  }
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

template <int ES>
__global__ void __cluster_dims__(kStCluster, 1, 1) __launch_bounds__(kStThreads)
    row_stats_kernel(const StatsProblem a) {
  constexpr int E = 16 / ES;                         // elements per vector
  constexpr int kRegEl = kStSlots * kStThreads * E;  // elements of a row segment in registers
  __shared__ StatsPart part;
  __shared__ float wred[4][kStWarps];
  __shared__ int wredi[2][kStWarps];
  __shared__ double wsum[kStWarps];
  __shared__ float merged[4];
  __shared__ int merged_flags;
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank());
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Kp = a.K > 0 ? a.K : 1;
  const int pair = static_cast<int>(blockIdx.x) / kStCluster;
  const int b = pair / Kp, i = pair % Kp;
  const float nanf = __int_as_float(0x7fc00000);

  // per-request arguments: the whole cluster takes the same branch
  const int nd = a.num_drafts ? a.num_drafts[b] : a.K;
  const float t = a.temperature[b];
  const int tk = a.top_k ? a.top_k[b] : 0;
  // a sampled request with a top-k filter takes its statistics from the
  // top-k lists (row_stats_topk_kernel); without lists it is an error
  const bool filtered = t > 0.f && tk > 0 && tk < a.V;
  if (filtered && tk <= a.max_topk && nd >= 0 && nd <= a.K) return;
  if (nd < 0 || nd > a.K || !(t >= 0.f) || tk < 0 || filtered) {
    if (i == 0 && rank == 0) {
      for (int j = tid; j < a.K; j += kStThreads) a.alpha[static_cast<size_t>(b) * a.K + j] = nanf;
      if (tid == 0) {
        a.expected[b] = nanf;
        record_error(&a.hdr->error, SV_DERR_ARG);
      }
    }
    return;
  }
  if (i >= nd) {
    if (rank == 0 && tid == 0) {
      if (i < a.K) a.alpha[static_cast<size_t>(b) * a.K + i] = nanf;
      if (nd == 0 && i == 0) a.expected[b] = 1.f;
    }
    return;
  }

  const char* prow = a.target + (static_cast<int64_t>(b) * (a.K + 1) + i) * a.t_stride;
  const char* qrow = a.draft + (static_cast<int64_t>(b) * a.K + i) * a.d_stride;
  const int seg = ((a.V + kStCluster - 1) / kStCluster + 7) & ~7;
  const int lo = min(a.V, rank * seg), hi = min(a.V, lo + seg);
  const int reg_hi = a.vec ? min(hi, lo + kRegEl) : lo;  // [lo, reg_hi) lives in registers
  const bool greedy = t == 0.f;
  const Scale2 c = scale_for(t);

  uint4 vp[kStSlots], vq[kStSlots];
#pragma unroll
  for (int k = 0; k < kStSlots; ++k) {
    const int e0 = lo + (tid + k * kStThreads) * E;
    if (e0 < reg_hi) {
      vp[k] = __ldcs(reinterpret_cast<const uint4*>(prow + static_cast<size_t>(e0) * ES));
      vq[k] = __ldcs(reinterpret_cast<const uint4*>(qrow + static_cast<size_t>(e0) * ES));
    } else {
      vp[k] = make_uint4(0u, 0u, 0u, 0u);
      vq[k] = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  // ---- pass 1: this CTA's (max, sum) of p and q, or their argmaxes
  int flags = 0;
  if (greedy) {
    float bv[2] = {kNegInf, kNegInf};
    int bi[2] = {0x7fffffff, 0x7fffffff};
    bool nan = false;
#pragma unroll
    for (int k = 0; k < kStSlots; ++k) {
      const int e0 = lo + (tid + k * kStThreads) * E;
      if (e0 < reg_hi) {
#pragma unroll
        for (int j = 0; j < E; ++j) {
          const float x = vec_elem<ES>(vp[k], j), y = vec_elem<ES>(vq[k], j);
          nan |= (x != x) | (y != y);
          if (x > bv[0]) { bv[0] = x; bi[0] = e0 + j; }
          if (y > bv[1]) { bv[1] = y; bi[1] = e0 + j; }
        }
      }
    }
    for (int e = reg_hi + tid; e < hi; e += kStThreads) {
      const float x = load_logit(prow, ES, e), y = load_logit(qrow, ES, e);
      nan |= (x != x) | (y != y);
      if (x > bv[0]) { bv[0] = x; bi[0] = e; }
      if (y > bv[1]) { bv[1] = y; bi[1] = e; }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const VI w = warp_reduce_vi(VI{bv[r], bi[r]});
      if (lane == 0) {
        wred[r][warp] = w.v;
        wredi[r][warp] = w.i;
      }
    }
    flags = __syncthreads_or(nan) ? SV_DERR_NONFINITE : 0;
    if (tid == 0) {
      VI r0{kNegInf, 0x7fffffff}, r1{kNegInf, 0x7fffffff};
      for (int w = 0; w < kStWarps; ++w) {
        r0 = vi_better(r0, VI{wred[0][w], wredi[0][w]});
        r1 = vi_better(r1, VI{wred[1][w], wredi[1][w]});
      }
      part.a0 = r0.v;
      part.a1 = __int_as_float(r0.i);
      part.a2 = r1.v;
      part.a3 = __int_as_float(r1.i);
      part.flags = flags;
      part.sum = 0.0;
    }
  } else {
    float m[2] = {kNegInf, kNegInf};
#pragma unroll
    for (int k = 0; k < kStSlots; ++k) {
      const int e0 = lo + (tid + k * kStThreads) * E;
      if (e0 < reg_hi) {
#pragma unroll
        for (int j = 0; j < E; ++j) {
          m[0] = max_nan(m[0], vec_elem<ES>(vp[k], j));
          m[1] = max_nan(m[1], vec_elem<ES>(vq[k], j));
        }
      }
    }
    for (int e = reg_hi + tid; e < hi; e += kStThreads) {
      m[0] = max_nan(m[0], load_logit(prow, ES, e));
      m[1] = max_nan(m[1], load_logit(qrow, ES, e));
    }
    const bool bad = (m[0] != m[0]) | (m[1] != m[1]) | (m[0] == kPosInf) | (m[1] == kPosInf);
    float s[2] = {0.f, 0.f};
    if (!bad) {
#pragma unroll
      for (int k = 0; k < kStSlots; ++k) {
        const int e0 = lo + (tid + k * kStThreads) * E;
        if (e0 < reg_hi) {
#pragma unroll
          for (int j = 0; j < E; ++j) {
            if (m[0] != kNegInf) s[0] += fast_exp2(scaled_arg(vec_elem<ES>(vp[k], j), m[0], c));
            if (m[1] != kNegInf) s[1] += fast_exp2(scaled_arg(vec_elem<ES>(vq[k], j), m[1], c));
          }
        }
      }
      for (int e = reg_hi + tid; e < hi; e += kStThreads) {
        if (m[0] != kNegInf) s[0] += fast_exp2(scaled_arg(load_logit(prow, ES, e), m[0], c));
        if (m[1] != kNegInf) s[1] += fast_exp2(scaled_arg(load_logit(qrow, ES, e), m[1], c));
      }
    }
    flags = __syncthreads_or(bad) ? SV_DERR_NONFINITE : 0;
    if (!flags) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const MS w = warp_reduce_ms(MS{m[r], s[r]}, c);
        if (lane == 0) {
          wred[2 * r][warp] = w.m;
          wred[2 * r + 1][warp] = w.s;
        }
      }
    }
    __syncthreads();
    if (tid == 0) {
      MS r0{kNegInf, 0.f}, r1{kNegInf, 0.f};
      if (!flags)
        for (int w = 0; w < kStWarps; ++w) {
          r0 = ms_combine(r0, MS{wred[0][w], wred[1][w]}, c);
          r1 = ms_combine(r1, MS{wred[2][w], wred[3][w]}, c);
        }
      part.a0 = r0.m;
      part.a1 = r0.s;
      part.a2 = r1.m;
      part.a3 = r1.s;
      part.flags = flags;
      part.sum = 0.0;
    }
  }

  // ---- exchange: every CTA merges the cluster's partials in rank order
  cl.sync();
  if (tid == 0) {
    int fl = 0;
    if (greedy) {
      VI r0{kNegInf, 0x7fffffff}, r1{kNegInf, 0x7fffffff};
      for (int r = 0; r < kStCluster; ++r) {
        const StatsPart* o = cl.map_shared_rank(&part, r);
        fl |= o->flags;
        r0 = vi_better(r0, VI{o->a0, __float_as_int(o->a1)});
        r1 = vi_better(r1, VI{o->a2, __float_as_int(o->a3)});
      }
      if (!fl && (r0.v == kPosInf || r1.v == kPosInf)) fl |= SV_DERR_NONFINITE;
      if (!fl && (r0.v == kNegInf || r1.v == kNegInf)) fl |= SV_DERR_MASS;
      merged[0] = r0.v;
      merged[1] = __int_as_float(r0.i);
      merged[2] = r1.v;
      merged[3] = __int_as_float(r1.i);
    } else {
      MS r0{kNegInf, 0.f}, r1{kNegInf, 0.f};
      for (int r = 0; r < kStCluster; ++r) {
        const StatsPart* o = cl.map_shared_rank(&part, r);
        fl |= o->flags;
        r0 = ms_combine(r0, MS{o->a0, o->a1}, c);
        r1 = ms_combine(r1, MS{o->a2, o->a3}, c);
      }
      if (!fl && !(r0.s > 0.f && r1.s > 0.f)) fl |= SV_DERR_MASS;
      merged[0] = r0.m;
      merged[1] = r0.s;
      merged[2] = r1.m;
      merged[3] = r1.s;
    }
    merged_flags = fl;
  }
  __syncthreads();
  const int fl = merged_flags;

  float alpha_val = nanf;
  if (greedy) {
    alpha_val = __float_as_int(merged[1]) == __float_as_int(merged[3]) ? 1.f : 0.f;
    cl.sync();  // no CTA leaves while another may still read its part
  } else {
    // ---- pass 2: sum of 2^min(a, b) over this CTA's segment
    float acc = 0.f;
    if (!fl) {
      const float mp = merged[0], mq = merged[2];
      const float lzp = static_cast<float>(log2(static_cast<double>(merged[1])));
      const float lzq = static_cast<float>(log2(static_cast<double>(merged[3])));
#pragma unroll
      for (int k = 0; k < kStSlots; ++k) {
        const int e0 = lo + (tid + k * kStThreads) * E;
        if (e0 < reg_hi) {
#pragma unroll
          for (int j = 0; j < E; ++j) {
            const float x = scaled_arg(vec_elem<ES>(vp[k], j), mp, c) - lzp;
            const float y = scaled_arg(vec_elem<ES>(vq[k], j), mq, c) - lzq;
            acc += fast_exp2(fminf(x, y));
          }
        }
      }
      for (int e = reg_hi + tid; e < hi; e += kStThreads) {
        const float x = scaled_arg(load_logit(prow, ES, e), mp, c) - lzp;
        const float y = scaled_arg(load_logit(qrow, ES, e), mq, c) - lzq;
        acc += fast_exp2(fminf(x, y));
      }
    }
    double d = static_cast<double>(acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (lane == 0) wsum[warp] = d;
    __syncthreads();
    if (tid == 0) {
      double sum = 0.0;
      for (int w = 0; w < kStWarps; ++w) sum += wsum[w];
      part.sum = sum;
    }
    cl.sync();
    if (rank == 0 && tid == 0 && !fl) {
      double sum = 0.0;
      for (int r = 0; r < kStCluster; ++r) sum += cl.map_shared_rank(&part, r)->sum;
      alpha_val = static_cast<float>(sum);
    }
    cl.sync();  // rank 0 has read every part
  }

  if (rank == 0 && tid == 0) {
    if (fl) {
      alpha_val = nanf;
      record_error(&a.hdr->error, fl);
    }
    a.alpha[static_cast<size_t>(b) * a.K + i] = alpha_val;
    __threadfence();
    const unsigned done = atomicAdd(a.tickets + b, 1u);
    if (done == static_cast<unsigned>(nd - 1)) {
      // the last position of the request: sum_{j<=nd} prod_{i<j} alpha_i
      __threadfence();
      double e = 0.0, reach = 1.0;
      for (int j = 0; j <= nd; ++j) {
        e += reach;
        if (j < nd) reach *= static_cast<double>(__ldcg(a.alpha + static_cast<size_t>(b) * a.K + j));
      }
      a.expected[b] = static_cast<float>(e);
      a.tickets[b] = 0u;
    }
  }
}

// Statistics of top-k requests from the top-k lists: row (b, i) of the lists
// is target row i for i <= nd and draft row i - nd - 1 after that, each its
// k largest logits in token order with (m, Z) over them (sv_topk.cuh).  One
// warp per request; p_i(x) = 2^((l - m) c) / Z on p_i's list and 0 off it,
// likewise q_i, so alpha_i = sum over the ids on both lists of min(p_i, q_i),
// in fp64.  Leaves the request's lists and (m, Z) zero, as the chain
// finalize does.
constexpr int kStTkWarps = 4;

struct StatsTopkProblem {
  int B, K, V, max_topk;
  bool has_draft;
  const int* num_drafts;
  const float* temperature;
  const int* top_k;
  float2* lists;  // [B (2K+1)][max_topk]
  float2* mz;     // [B (2K+1)]
  float* alpha;
  float* expected;
  WsHeader* hdr;
};

__global__ void __launch_bounds__(kStTkWarps * 32) row_stats_topk_kernel(const StatsTopkProblem a) {
  __shared__ int q_ids[kStTkWarps][SV_MAX_TOPK];
  __shared__ float q_val[kStTkWarps][SV_MAX_TOPK];
  grid_dependency_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = static_cast<int>(blockIdx.x) * kStTkWarps + warp;
  if (b >= a.B) return;
  const int nd = a.num_drafts ? a.num_drafts[b] : a.K;
  const float t = a.temperature[b];
  const int k = a.top_k ? a.top_k[b] : 0;
  if (chain_kind(nd, t, k, a.K, a.V, a.max_topk, a.has_draft) != KIND_TOPK) return;
  const int R = 2 * a.K + 1;
  const size_t r0 = static_cast<size_t>(b) * R;
  const int nrows = 2 * nd + 1;
  const Scale2 c = scale_for(t);
  const double cd = static_cast<double>(c.hi) + static_cast<double>(c.lo);
  int err = 0;
  for (int j = lane; j < nrows; j += 32) {
    const float2 v = a.mz[r0 + j];
    if (v.x != v.x) err |= SV_DERR_NONFINITE;
    else if (v.x == kNegInf || !(v.y > 0.f)) err |= SV_DERR_MASS;
  }
  err = __reduce_or_sync(0xffffffffu, err);
  double e = 1.0, reach = 1.0;
  for (int i = 0; i < nd && !err; ++i) {
    const float2* pl = a.lists + (r0 + i) * a.max_topk;
    const float2* ql = a.lists + (r0 + nd + 1 + i) * a.max_topk;
    const float2 mzp = a.mz[r0 + i], mzq = a.mz[r0 + nd + 1 + i];
    for (int s = lane; s < k; s += 32) {
      const float2 v = ql[s];
      q_ids[warp][s] = __float_as_int(v.y);
      q_val[warp][s] = v.x;
    }
    __syncwarp();
    double acc = 0.0;
    for (int s = lane; s < k; s += 32) {
      const float2 v = pl[s];
      const int id = __float_as_int(v.y);
      // q's list is in token order: binary search for id
      int lo = 0, hi = k - 1, at = -1;
      while (lo <= hi && id >= 0) {
        const int mid = (lo + hi) >> 1;
        const int qm = q_ids[warp][mid];
        if (qm == id) {
          at = mid;
          break;
        }
        if (qm < id) lo = mid + 1;
        else hi = mid - 1;
      }
      if (at >= 0) {
        const double pp = exp2_nonpos((static_cast<double>(v.x) - mzp.x) * cd) / mzp.y;
        const double qq = exp2_nonpos((static_cast<double>(q_val[warp][at]) - mzq.x) * cd) / mzq.y;
        acc += pp < qq ? pp : qq;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) a.alpha[static_cast<size_t>(b) * a.K + i] = static_cast<float>(acc);
    reach *= acc;
    e += reach;
    __syncwarp();
  }
  if (lane == 0) {
    if (err) {
      for (int i = 0; i < a.K; ++i) a.alpha[static_cast<size_t>(b) * a.K + i] = __int_as_float(0x7fc00000);
      a.expected[b] = __int_as_float(0x7fc00000);
      record_error(&a.hdr->error, err);
    } else {
      for (int i = nd; i < a.K; ++i) a.alpha[static_cast<size_t>(b) * a.K + i] = __int_as_float(0x7fc00000);
      a.expected[b] = static_cast<float>(e);
    }
  }
  // leave the lists and (m, Z) of the request's rows zero
  for (int j = 0; j < nrows; ++j) {
    float2* l = a.lists + (r0 + j) * a.max_topk;
    for (int s = lane; s < a.max_topk; s += 32) l[s] = make_float2(0.f, 0.f);
  }
  for (int j = lane; j < nrows; j += 32) a.mz[r0 + j] = make_float2(0.f, 0.f);
}

}  // namespace sv
