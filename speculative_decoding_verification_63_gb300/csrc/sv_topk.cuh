// sv_topk.cuh -- the top-k lists of filtered rows, a pass of its own that
// runs before the persistent kernel.
//
// With top-k filtering, p and q are each restricted to their own k most
// likely tokens before the accept tests and the residual ("LLM speculative
// decoding study notes 02", sec. 5.4: the draft and the target decode with
// the same strategy; the kept set is the k largest logits, ties at the k-th
// value going to the lower token id).  Neither the accept tests nor the
// residual then need the row again: they need the kept (logit, id) pairs
// and the row's (m, Z) over them.  This pass produces exactly that, per
// filtered row, in three steps that need no barrier between warps:
//
//   segment  a row is cut into S segments of seg_len tokens; one warp
//            streams a segment once, keeping candidates in its own shared
//            buffer: every element at first, then only elements whose key
//            is above the k-th best key so far (later elements have
//            higher ids, so an equal key ranks lower and cannot enter).
//            When the buffer fills it is cut to its exact top-k.  The
//            buffer is kept in token order throughout.
//   publish  the warp writes its segment's top-k (token order) and count,
//            fences, and bumps the row's counter;
//   merge    the warp that brings the counter to S concatenates the S lists
//            (segment order = token order), cuts them to the row's exact
//            top-k, writes the list and (m, Z) and zeroes the counter.
//
// Keys are order-preserving unsigned integers of the logit bits (16-bit
// for bf16, 32-bit for fp32), 0 for NaN and for padding; -0 counts as +0,
// so equal logits have equal keys.  An exact cut finds the k-th largest key
// K* by bisection over the key range, keeps the keys above K*, and the
// first (lowest-id) entries equal to K* up to k in all.
#pragma once

#include "sv_rowpass.cuh"

namespace sv {

constexpr int kTkWarps = 8;     // warps per CTA
constexpr int kTkCtasPerSm = 3; // resident CTAs per SM (launch bounds): the grid is one wave
constexpr int kTkThreads = kTkWarps * 32;
constexpr int kTkCap = 512;     // candidates a warp holds
constexpr int kTkMaxSegs = 8;   // segments per row (kTkMaxSegs * SV_MAX_TOPK <= kTkCap)
constexpr int kTkStep = 256;    // tokens per warp step (8 per lane)
constexpr int kTkUnroll = 4;    // steps whose loads are in flight together
constexpr int kTkMinSeg = 8192; // a row is cut into ceil(V / kTkMinSeg) segments, at most 8

struct TopkPass {
  int n_req, K, V, es, max_topk;
  int n_seg, seg_len;        // segments per row, tokens per segment (multiple of kTkStep)
  bool vec;                  // row starts and strides are 16-byte aligned
  bool has_draft;
  const char* target;
  int64_t t_stride;          // bytes
  const char* draft;
  int64_t d_stride;
  const int* num_drafts;
  const float* temperature;
  const int* top_k;
  float2* seg_lists;         // [B (2K+1) n_seg][max_topk] (logit, id bits), token order
  int* seg_count;            // [B (2K+1) n_seg] entries kept; -1: NaN or +inf seen
  float2* lists;             // [B (2K+1)][max_topk] the row's top-k, token order, padded
                             // with (-inf, -1)
  float2* mz;                // [B (2K+1)] (m, Z) over the kept logits; (NaN, 0) for a row
                             // with NaN or +inf
  unsigned* row_done;        // [B (2K+1)] segments published (zero between calls)
};

// Order-preserving keys.  bf16: x is the 16-bit pattern; fp32: the 32-bit
// pattern.  NaN -> 0; -0 -> the key of +0.
__device__ __forceinline__ unsigned tk_key16(unsigned x) {
  if (x == 0x8000u) x = 0u;
  if ((x & 0x7fffu) > 0x7f80u) return 0u;
  return (x & 0x8000u) ? (~x & 0xffffu) : (x | 0x8000u);
}
__device__ __forceinline__ unsigned tk_key32(unsigned x) {
  if (x == 0x80000000u) x = 0u;
  if ((x & 0x7fffffffu) > 0x7f800000u) return 0u;
  return (x & 0x80000000u) ? ~x : (x | 0x80000000u);
}
// the logit of a key (key != 0)
__device__ __forceinline__ float tk_value(unsigned key, int es) {
  if (es == 2) {
    const unsigned h = (key & 0x8000u) ? (key & 0x7fffu) : (~key & 0xffffu);
    return __uint_as_float(h << 16);
  }
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}
__device__ __forceinline__ unsigned tk_key_of(float v, int es) {
  return es == 2 ? tk_key16(__float_as_uint(v) >> 16) : tk_key32(__float_as_uint(v));
}

// One warp's candidate buffer (shared memory) and its state.  The state is
// the same in every lane (all updates are warp-wide).
struct TkBuf {
  unsigned* key;
  int* id;
  int cnt;        // entries held, token order
  bool have;      // thr holds the k-th best key of everything seen
  unsigned thr;
};

__device__ __forceinline__ unsigned tk_count_ge(const TkBuf& bf, unsigned t, int lane) {
  unsigned c = 0;
  for (int i = lane; i < bf.cnt; i += 32) c += bf.key[i] >= t ? 1u : 0u;
  return __reduce_add_sync(0xffffffffu, c);
}

// Cut the buffer to its exact top-k (k >= 1), in place and in token order.
__device__ void tk_cut(TkBuf& bf, int k, int lane) {
  __syncwarp();
  if (bf.cnt <= k) {
    if (bf.cnt == k) {  // the k-th best is the smallest key held
      unsigned mn = 0xffffffffu;
      for (int i = lane; i < bf.cnt; i += 32) mn = min(mn, bf.key[i]);
      bf.thr = __reduce_min_sync(0xffffffffu, mn);
      bf.have = true;
    }
    return;
  }
  unsigned mx = 0;
  for (int i = lane; i < bf.cnt; i += 32) mx = max(mx, bf.key[i]);
  mx = __reduce_max_sync(0xffffffffu, mx);
  // K*: the largest t with at least k keys >= t (keys of held entries >= 1)
  unsigned lo = 1u, hi = mx;
  while (lo < hi) {
    const unsigned mid = lo + (hi - lo + 1u) / 2u;
    if (tk_count_ge(bf, mid, lane) >= static_cast<unsigned>(k)) lo = mid;
    else hi = mid - 1u;
  }
  const unsigned kstar = lo;
  const unsigned gt = tk_count_ge(bf, kstar + 1u, lane);  // < k
  const unsigned need = static_cast<unsigned>(k) - gt;     // entries equal to K* to keep
  const unsigned lt_mask = (1u << lane) - 1u;
  unsigned written = 0, ties = 0;
  for (int base = 0; base < bf.cnt; base += 32) {
    const int i = base + lane;
    const bool in = i < bf.cnt;
    const unsigned key = in ? bf.key[i] : 0u;
    const int id = in ? bf.id[i] : 0;
    const bool tie = in && key == kstar;
    const unsigned tmask = __ballot_sync(0xffffffffu, tie);
    const bool keep = in && (key > kstar || (tie && ties + __popc(tmask & lt_mask) < need));
    const unsigned kmask = __ballot_sync(0xffffffffu, keep);
    __syncwarp();  // every lane has read its entry of this tile
    if (keep) {
      const unsigned p = written + __popc(kmask & lt_mask);  // <= i: never ahead of a read
      bf.key[p] = key;
      bf.id[p] = id;
    }
    written += __popc(kmask);
    ties += __popc(tmask);
    __syncwarp();
  }
  bf.cnt = static_cast<int>(written);
  bf.thr = kstar;
  bf.have = true;
}

// Keys of the 8 tokens e .. e+7 of a segment of n tokens (0 past n), and
// whether one of them is NaN or +inf.
template <int ES>
__device__ __forceinline__ void tk_keys_scalar(const char* seg, int e, int n, unsigned (&key)[8],
                                               bool& bad) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    key[j] = 0u;
    if (e + j < n) {
      if constexpr (ES == 2) {
        const unsigned x = reinterpret_cast<const unsigned short*>(seg)[e + j];
        bad |= (x & 0x7fffu) >= 0x7f80u && x != 0xff80u;
        key[j] = tk_key16(x);
      } else {
        const unsigned x = reinterpret_cast<const unsigned*>(seg)[e + j];
        bad |= (x & 0x7fffffffu) >= 0x7f800000u && x != 0xff800000u;
        key[j] = tk_key32(x);
      }
    }
  }
}

template <int ES>
__device__ __forceinline__ void tk_keys_vec(const uint4 (&r)[ES / 2], unsigned (&key)[8],
                                            bool& bad) {
  if constexpr (ES == 2) {
    const unsigned w[4] = {r[0].x, r[0].y, r[0].z, r[0].w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const unsigned lo = w[h] & 0xffffu, hi = w[h] >> 16;
      bad |= ((lo & 0x7fffu) >= 0x7f80u && lo != 0xff80u) ||
             ((hi & 0x7fffu) >= 0x7f80u && hi != 0xff80u);
      key[2 * h] = tk_key16(lo);
      key[2 * h + 1] = tk_key16(hi);
    }
  } else {
    const unsigned w[8] = {r[0].x, r[0].y, r[0].z, r[0].w, r[1].x, r[1].y, r[1].z, r[1].w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      bad |= (w[j] & 0x7fffffffu) >= 0x7f800000u && w[j] != 0xff800000u;
      key[j] = tk_key32(w[j]);
    }
  }
}

// Append the passing keys of one step (token ids id0 + 8 lane + j) to the
// buffer, cutting it first if they would not fit.
__device__ __forceinline__ void tk_append(TkBuf& bf, const unsigned (&key)[8], int id0, int k,
                                          int lane) {
  unsigned pass = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) pass |= (bf.have ? key[j] > bf.thr : key[j] != 0u) ? (1u << j) : 0u;
  unsigned c = __popc(pass);
  unsigned total = __reduce_add_sync(0xffffffffu, c);
  if (total == 0u) return;
  if (bf.cnt + static_cast<int>(total) > kTkCap) {
    tk_cut(bf, k, lane);  // now cnt <= k, have: the step is filtered again
    pass = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) pass |= key[j] > bf.thr ? (1u << j) : 0u;
    c = __popc(pass);
    total = __reduce_add_sync(0xffffffffu, c);
    if (total == 0u) return;
  }
  const unsigned incl = warp_incl_scan_u(c, lane);
  unsigned slot = static_cast<unsigned>(bf.cnt) + incl - c;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (pass & (1u << j)) {
      bf.key[slot] = key[j];
      bf.id[slot] = id0 + 8 * lane + j;
      ++slot;
    }
  bf.cnt += static_cast<int>(total);
  __syncwarp();
  if (!bf.have && bf.cnt >= k) tk_cut(bf, k, lane);
}

// One segment: tokens [s0, s0 + n) of a row.
template <int ES>
__device__ void tk_segment(const TopkPass& a, const char* row, int s0, int n, int k, TkBuf& bf,
                           bool& bad, int lane) {
  constexpr int U = kTkUnroll * 2 / ES;  // the same bytes in flight for bf16 and fp32
  const char* seg = row + static_cast<size_t>(s0) * ES;
  for (int e0 = 0; e0 < n; e0 += kTkStep * U) {
    uint4 raw[U][ES / 2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = e0 + u * kTkStep + 8 * lane;
      if (a.vec && e + 8 <= n) {
        const uint4* p = reinterpret_cast<const uint4*>(seg + static_cast<size_t>(e) * ES);
#pragma unroll
        for (int h = 0; h < ES / 2; ++h) raw[u][h] = __ldcs(p + h);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int eb = e0 + u * kTkStep;
      if (eb >= n) break;  // warp-uniform
      unsigned key[8];
      const int e = eb + 8 * lane;
      if (a.vec && e + 8 <= n) tk_keys_vec<ES>(raw[u], key, bad);
      else tk_keys_scalar<ES>(seg, e, n, key, bad);
      tk_append(bf, key, s0 + eb, k, lane);
    }
  }
}

// The warp that published a row's last segment: merge the row.
__device__ void tk_merge(const TopkPass& a, int r, int k, Scale2 c, TkBuf& bf, int lane) {
  bool bad = false;
  bf.cnt = 0;
  bf.have = false;
  for (int s = 0; s < a.n_seg; ++s) {
    // a segment keeps at most k entries (the clamp only guards the buffer)
    const int ns = min(__ldcg(a.seg_count + static_cast<size_t>(r) * a.n_seg + s), k);
    if (ns < 0) {
      bad = true;
      continue;
    }
    const float2* src = a.seg_lists + (static_cast<size_t>(r) * a.n_seg + s) * a.max_topk;
    for (int i = lane; i < ns; i += 32) {
      const float2 v = __ldcg(src + i);
      bf.key[bf.cnt + i] = tk_key_of(v.x, a.es);
      bf.id[bf.cnt + i] = __float_as_int(v.y);
    }
    bf.cnt += ns;
  }
  __syncwarp();
  // leave the row's segment lists and counts zero for the next call (any
  // part of the workspace may serve another call's partials, which must
  // start at zero)
  for (int s = 0; s < a.n_seg; ++s) {
    float2* src = a.seg_lists + (static_cast<size_t>(r) * a.n_seg + s) * a.max_topk;
    for (int i = lane; i < a.max_topk; i += 32) src[i] = make_float2(0.f, 0.f);
    if (lane == 0) a.seg_count[static_cast<size_t>(r) * a.n_seg + s] = 0;
  }
  if (bf.cnt > k) tk_cut(bf, k, lane);
  __syncwarp();
  float2* out = a.lists + static_cast<size_t>(r) * a.max_topk;
  float m = kNegInf;
  for (int i = lane; i < k; i += 32) {
    const bool in = i < bf.cnt;
    const float v = in ? tk_value(bf.key[i], a.es) : kNegInf;
    out[i] = make_float2(v, __int_as_float(in ? bf.id[i] : -1));
    m = fmaxf(m, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = 0.f;
  if (m != kNegInf)
    for (int i = lane; i < bf.cnt; i += 32) z += fast_exp2(scaled_arg(tk_value(bf.key[i], a.es), m, c));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane == 0) {
    a.mz[r] = bad ? make_float2(__int_as_float(0x7fc00000), 0.f) : make_float2(m, z);
    a.row_done[r] = 0u;  // ready for the next call
  }
  __syncwarp();
}

__global__ void __launch_bounds__(kTkThreads, kTkCtasPerSm) topk_kernel(const TopkPass a) {
  __shared__ unsigned s_key[kTkWarps][kTkCap];
  __shared__ int s_id[kTkWarps][kTkCap];
  grid_dependency_wait();
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = 2 * a.K + 1;
  const int n_items = a.n_req * R * a.n_seg;
  const int gw = blockIdx.x * kTkWarps + warp;
  const int W = gridDim.x * kTkWarps;
  for (int item = gw; item < n_items; item += W) {
    const int r = item / a.n_seg, s = item % a.n_seg;
    const int b = r / R, rl = r % R;
    const int nd = a.num_drafts ? a.num_drafts[b] : a.K;
    const float t = a.temperature[b];
    const int k = a.top_k ? a.top_k[b] : 0;
    if (chain_kind(nd, t, k, a.K, a.V, a.max_topk, a.has_draft) != KIND_TOPK || rl > 2 * nd)
      continue;
    const char* row = rl <= nd
        ? a.target + (static_cast<int64_t>(b) * (a.K + 1) + rl) * a.t_stride
        : a.draft + (static_cast<int64_t>(b) * a.K + (rl - nd - 1)) * a.d_stride;
    const int s0 = s * a.seg_len;
    const int n = min(a.seg_len, a.V - s0);
    TkBuf bf{s_key[warp], s_id[warp], 0, false, 0u};
    bool bad = false;
    if (a.es == 2) tk_segment<2>(a, row, s0, n, k, bf, bad, lane);
    else tk_segment<4>(a, row, s0, n, k, bf, bad, lane);
    bad = __any_sync(0xffffffffu, bad);
    if (bf.cnt > k) tk_cut(bf, k, lane);
    __syncwarp();
    float2* dst = a.seg_lists + static_cast<size_t>(item) * a.max_topk;
    for (int i = lane; i < bf.cnt; i += 32) dst[i] = make_float2(tk_value(bf.key[i], a.es), __int_as_float(bf.id[i]));
    if (lane == 0) a.seg_count[item] = bad ? -1 : bf.cnt;
    __syncwarp();
    __threadfence();  // the segment's list and count before the row counter
    unsigned old = 0;
    if (lane == 0) old = atomicAdd(a.row_done + r, 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old + 1u == static_cast<unsigned>(a.n_seg)) {
      __threadfence();  // the other segments' lists, published before their increments
      const Scale2 c = scale_for(t);
      tk_merge(a, r, k, c, bf, lane);
    }
  }
}

}  // namespace sv
